// k_quant.cu -- Q8_0 activation quantiser, int4 weight converter, and the
// stage kernel for per-block integer dot products.
//
// Q8_0 ("colibri: a pure-C inference engine ...", discuss.pytorch.kr, section
// "Key features"; "Open-source engine that ran 744B GLM-5.2 ...", jeff.news,
// section "Attention and kernels"): blocks of 32, amax/127 F32 scale, codes by
// round-half-even.  The int4 container ("GLM-5.2-colibri-int4" model card,
// sections "TL;DR" and "Technical features"): per-row F32 scale max|w|/7,
// codes clamp(rint(w/s), -7, 7) stored as nibbles q+8, low nibble first.
#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

// One warp per block of 32 activations; lane i owns element i.
__global__ void __launch_bounds__(256) k_q8_0(const float *__restrict__ x, long nblocks,
                                              int8_t *__restrict__ q, float *__restrict__ d)
{
    long blk = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (blk >= nblocks) return;
    float v = x[blk * 32 + lane];
    float db;
    int qi = q8_0_lane(v, &db);
    q[blk * 32 + lane] = (int8_t)qi;
    if (lane == 0) d[blk] = db;
}

// One warp per weight row.
__global__ void __launch_bounds__(256) k_pack_int4(const float *__restrict__ w, int rows, int K,
                                                   uint8_t *__restrict__ packed,
                                                   float *__restrict__ scale)
{
    int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *wr = w + (size_t)row * K;
    float a = 0.0f;
    for (int k = lane; k < K; k += 32) a = fmaxf(a, fabsf(wr[k]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(FULL, a, o));
    float s = __fdiv_rn(a, 7.0f);
    if (lane == 0) scale[row] = s;
    uint8_t *pr = packed + (size_t)row * (K / 2);
    for (int j = lane; j < K / 2; j += 32) {
        float2 v = reinterpret_cast<const float2 *>(wr)[j];
        int q0 = 0, q1 = 0;
        if (s > 0.0f) {
            q0 = max(-7, min(7, __float2int_rn(__fdiv_rn(v.x, s))));
            q1 = max(-7, min(7, __float2int_rn(__fdiv_rn(v.y, s))));
        }
        pr[j] = (uint8_t)((q0 + 8) | ((q1 + 8) << 4));
    }
}

// The int8 weight container, one warp per row: s = max|row| / 127 (IEEE
// divide), q = clamp(rint(w / s), -127, 127) as two's-complement bytes; an
// all-zero row gives s = 0 and codes 0.  The same rule as the int4 container
// with 127 in place of 7 (the pages name an int8 container and an int8 head:
// "colibri: a pure-C inference engine ..." (discuss.pytorch.kr), section
// "Key features").
__global__ void __launch_bounds__(256) k_pack_int8(const float *__restrict__ w, int rows, int K,
                                                   int8_t *__restrict__ q, float *__restrict__ scale)
{
    int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *wr = w + (size_t)row * K;
    float a = 0.0f;
    for (int k = lane; k < K; k += 32) a = fmaxf(a, fabsf(wr[k]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(FULL, a, o));
    float s = __fdiv_rn(a, 127.0f);
    if (lane == 0) scale[row] = s;
    int8_t *qr = q + (size_t)row * K;
    for (int k = lane; k < K; k += 32) {
        int v = 0;
        if (s > 0.0f) v = max(-127, min(127, __float2int_rn(__fdiv_rn(wr[k], s))));
        qr[k] = (int8_t)v;
    }
}

// Stage kernel: I[r][b] of int8-container rows against one int8 vector.
__global__ void __launch_bounds__(256) k_block_dots_w8(const int8_t *__restrict__ w8, int rows, int K,
                                                       const int8_t *__restrict__ q, int32_t *__restrict__ I)
{
    int nb = K / 32;
    long id = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (long)rows * nb) return;
    int r = (int)(id / nb), b = (int)(id % nb);
    const int4 *xq = reinterpret_cast<const int4 *>(q + (size_t)b * 32);
    const int4 *wq = reinterpret_cast<const int4 *>(w8 + (size_t)r * K + (size_t)b * 32);
    int acc = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int4 x = xq[h], w = wq[h];
        acc = __dp4a(w.x, x.x, acc);
        acc = __dp4a(w.y, x.y, acc);
        acc = __dp4a(w.z, x.z, acc);
        acc = __dp4a(w.w, x.w, acc);
    }
    I[id] = acc;
}

// Stage kernel: I[r][b] for packed rows against one int8 vector, through the
// same block_dot used by the expert kernels.  One thread per (row, block).
__global__ void __launch_bounds__(256) k_block_dots(const uint8_t *__restrict__ w4, int rows, int K,
                                                    const int8_t *__restrict__ q,
                                                    int32_t *__restrict__ I)
{
    int nb = K / 32;
    long id = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (long)rows * nb) return;
    int r = (int)(id / nb), b = (int)(id % nb);
    const uint4 *xq = reinterpret_cast<const uint4 *>(q + (size_t)b * 32);
    uint4 lo, hi;
    int sum;
    split_block(xq[0], xq[1], &lo, &hi, &sum);
    uint4 w = *reinterpret_cast<const uint4 *>(w4 + (size_t)r * (K / 2) + (size_t)b * 16);
    I[id] = block_dot(w, lo, hi, -8 * sum);
}

int launch_q8_0(const float *x, long n, int8_t *q, float *d, cudaStream_t st)
{
    long nblocks = n / 32;
    if (nblocks == 0) return 0;
    long threads = nblocks * 32;
    unsigned grid = (unsigned)((threads + 255) / 256);
    k_q8_0<<<grid, 256, 0, st>>>(x, nblocks, q, d);
    count_launch();
    return 0;
}

int launch_pack_int4(const float *w, int rows, int K, uint8_t *packed, float *scale, cudaStream_t st)
{
    if (rows == 0) return 0;
    unsigned grid = (unsigned)(((long)rows * 32 + 255) / 256);
    k_pack_int4<<<grid, 256, 0, st>>>(w, rows, K, packed, scale);
    count_launch();
    return 0;
}

int launch_pack_int8(const float *w, int rows, int K, int8_t *q, float *scale, cudaStream_t st)
{
    if (rows == 0) return 0;
    unsigned grid = (unsigned)(((long)rows * 32 + 255) / 256);
    k_pack_int8<<<grid, 256, 0, st>>>(w, rows, K, q, scale);
    count_launch();
    return 0;
}

int launch_block_dots_w8(const int8_t *w8, int rows, int K, const int8_t *q, int32_t *I, cudaStream_t st)
{
    long n = (long)rows * (K / 32);
    if (n == 0) return 0;
    k_block_dots_w8<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w8, rows, K, q, I);
    count_launch();
    return 0;
}

int launch_block_dots(const uint8_t *w4, int rows, int K, const int8_t *q, int32_t *I, cudaStream_t st)
{
    long n = (long)rows * (K / 32);
    if (n == 0) return 0;
    k_block_dots<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w4, rows, K, q, I);
    count_launch();
    return 0;
}

}  // namespace coli

namespace coli {

// ---------------------------------------------------------------------------
// Pre-norm of a stacked decoder layer: xn = x / sqrt(mean(x^2) + eps) per
// token, no learned gain.  The sum of squares follows the router logits' fixed
// order (chunks of 4 into 256 partials, chunks ascending, one fma per element;
// xor-butterfly folds over 32 and then 8), and the scalar steps are single
// IEEE operations, so the result is reproducible bit for bit.  One block of
// 256 threads per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rmsnorm(const float *__restrict__ x, int H, float eps,
                                                 float *__restrict__ xn)
{
    const int t = blockIdx.x, j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const float4 *xt = reinterpret_cast<const float4 *>(x + (size_t)t * H);
    float p = 0.0f;
    for (int c = j; c < (H >> 2); c += 256) {
        const float4 v = __ldg(xt + c);
        p = __fmaf_rn(v.x, v.x, p);
        p = __fmaf_rn(v.y, v.y, p);
        p = __fmaf_rn(v.z, v.z, p);
        p = __fmaf_rn(v.w, v.w, p);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(FULL, p, o));
    __shared__ float red[8];
    __shared__ float r_sh;
    if (lane == 0) red[warp] = p;
    __syncthreads();
    if (j == 0) {
        float s[8], tmp[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) s[w] = red[w];
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
#pragma unroll
            for (int w = 0; w < 8; ++w) tmp[w] = __fadd_rn(s[w], s[w ^ o]);
#pragma unroll
            for (int w = 0; w < 8; ++w) s[w] = tmp[w];
        }
        const float ms = __fdiv_rn(s[0], (float)H);
        r_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();
    const float r = r_sh;
    float4 *ot = reinterpret_cast<float4 *>(xn + (size_t)t * H);
    for (int c = j; c < (H >> 2); c += 256) {
        const float4 v = __ldg(xt + c);
        ot[c] = make_float4(__fmul_rn(v.x, r), __fmul_rn(v.y, r), __fmul_rn(v.z, r), __fmul_rn(v.w, r));
    }
}

int launch_rmsnorm(const float *x, int T, int H, float eps, float *xn, cudaStream_t st)
{
    if (T <= 0) return 0;
    k_rmsnorm<<<T, 256, 0, st>>>(x, H, eps, xn);
    count_launch();
    return 0;
}

}  // namespace coli
