// coli_common.cuh -- device helpers shared by the layer's kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle: the two are written separately
// from the method's definition.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace coli {

constexpr unsigned FULL = 0xffffffffu;

// Device status word bits (read back by coli_moe_get_device_status).
constexpr int ST_BAD_INDEX = 1;   // an expert index outside [0, E)
constexpr int ST_TIMEOUT = 2;     // a bounded wait gave up
constexpr int ST_BAD_SHAPE = 4;   // a kernel met a shape (or a shared-memory base) it does not support

// Tokens per GEMV tile: one pass over an expert's weights serves up to this
// many of the tokens routed to it.
constexpr int GEMV_MT = 4;

// ---------------------------------------------------------------------------
// Own exponential and sigmoid.  Cody-Waite reduction z = n ln2 + r with
// n = rint(z log2 e) and a two-part ln2, e^r by its Taylor series to degree 7,
// times 2^n built from exponent bits (W. J. Cody, W. Waite, "Software Manual
// for the Elementary Functions", 1980).  Written with explicit round-to-nearest
// operations so that no contraction or reassociation changes the result: the
// router's expert choice must be reproducible bit for bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float own_exp(float z)
{
    if (z > 88.0f) return __int_as_float(0x7f800000);
    if (z < -87.0f) return 0.0f;
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e430p-1f;
    const float ln2_lo = -0x1.05c610p-29f;
    float t = __fmul_rn(z, log2e);
    float n = rintf(t);
    float r = __fmaf_rn(-n, ln2_hi, z);
    r = __fmaf_rn(-n, ln2_lo, r);
    // 1/k! for k = 7 .. 0, rounded to F32
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1.000000p-1f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    int ni = (int)n;
    float two_n = __int_as_float((ni + 127) << 23);
    return __fmul_rn(p, two_n);
}

// sigma(z) = 1 / (1 + e^-z)
__device__ __forceinline__ float own_sigmoid(float z)
{
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, own_exp(-z)));
}

// ---------------------------------------------------------------------------
// Q8_0 of one value inside a warp-wide block of 32 (lane i holds element i).
// amax = max|x|, d = amax / 127, q = clamp(rint(x * (1/d)), -127, 127).
// Returns the code; *d_out receives d on every lane.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int q8_0_lane(float v, float *d_out)
{
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(FULL, a, o));
    float d = __fdiv_rn(a, 127.0f);
    float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    int q = __float2int_rn(__fmul_rn(v, id));
    q = max(-127, min(127, q));
    *d_out = d;
    return q;
}

// ---------------------------------------------------------------------------
// Integer dot of one 32-wide block: 16 bytes of packed nibbles (element 2j in
// the low nibble of byte j) against 32 int8 activations held in "split" form:
// xlo word g = elements (8g, 8g+2, 8g+4, 8g+6), xhi word g = (8g+1, 8g+3,
// 8g+5, 8g+7).  The masked low nibbles of weight word g line up with xlo word
// g and the shifted high nibbles with xhi word g, so no byte shuffling of the
// weights is needed.  Returns c + sum(nibble * x); the -8 nibble offset is
// folded into c by the caller (c = ... - 8 * sum(x)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int block_dot(uint4 w, uint4 xlo, uint4 xhi, int c)
{
    c = dp4a_us(w.x & 0x0F0F0F0Fu, (int)xlo.x, c);
    c = dp4a_us((w.x >> 4) & 0x0F0F0F0Fu, (int)xhi.x, c);
    c = dp4a_us(w.y & 0x0F0F0F0Fu, (int)xlo.y, c);
    c = dp4a_us((w.y >> 4) & 0x0F0F0F0Fu, (int)xhi.y, c);
    c = dp4a_us(w.z & 0x0F0F0F0Fu, (int)xlo.z, c);
    c = dp4a_us((w.z >> 4) & 0x0F0F0F0Fu, (int)xhi.z, c);
    c = dp4a_us(w.w & 0x0F0F0F0Fu, (int)xlo.w, c);
    c = dp4a_us((w.w >> 4) & 0x0F0F0F0Fu, (int)xhi.w, c);
    return c;
}

// Split 32 natural-order int8 codes (two uint4) into the xlo / xhi form above
// and return their sum.
__device__ __forceinline__ void split_block(uint4 a, uint4 b, uint4 *lo, uint4 *hi, int *sum)
{
    // natural words: a.x = e0..3, a.y = e4..7, a.z = e8..11, a.w = e12..15, b = e16..31
    lo->x = __byte_perm(a.x, a.y, 0x6420);
    hi->x = __byte_perm(a.x, a.y, 0x7531);
    lo->y = __byte_perm(a.z, a.w, 0x6420);
    hi->y = __byte_perm(a.z, a.w, 0x7531);
    lo->z = __byte_perm(b.x, b.y, 0x6420);
    hi->z = __byte_perm(b.x, b.y, 0x7531);
    lo->w = __byte_perm(b.z, b.w, 0x6420);
    hi->w = __byte_perm(b.z, b.w, 0x7531);
    int s = 0;
    s = __dp4a((int)a.x, 0x01010101, s);
    s = __dp4a((int)a.y, 0x01010101, s);
    s = __dp4a((int)a.z, 0x01010101, s);
    s = __dp4a((int)a.w, 0x01010101, s);
    s = __dp4a((int)b.x, 0x01010101, s);
    s = __dp4a((int)b.y, 0x01010101, s);
    s = __dp4a((int)b.z, 0x01010101, s);
    s = __dp4a((int)b.w, 0x01010101, s);
    *sum = s;
}

// int32 -> F32 by the exponent trick: bit pattern 0x4B400000 + I is the float
// 12582912 + I for |I| < 2^22, so subtracting 12582912 gives I exactly.
constexpr int MAGIC_I = 0x4B400000;
constexpr float MAGIC_F = 12582912.0f;

__device__ __forceinline__ void set_status(int *status, int bit)
{
    if (status) atomicOr(status, bit);
}

}  // namespace coli
