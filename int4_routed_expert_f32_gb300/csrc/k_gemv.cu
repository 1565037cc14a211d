// k_gemv.cu -- expert matmuls for decode-sized batches: int4 x int8 streaming
// GEMV with dp4a, per-block int32 dot products scaled in F32, the SiLU*up
// product and Q8_0 requantisation of the hidden fused into the gate/up
// epilogue, then the down GEMV, then the gate-weighted combine.
//
// Method: int8 (Q8_0-style) activations against packed int4 weights with an
// integer dot product per block ("colibri: a pure-C inference engine ...",
// discuss.pytorch.kr, section "Key features"; "Colibri: an AI engine running a
// 744B model in 25GB of RAM", alphamatch.ai, section "Optimised integer
// kernels"); SwiGLU experts plus a shared expert ("Open-source engine that ran
// 744B GLM-5.2 on a 25GB-RAM laptop", jeff.news, section "Attention and
// kernels").
//
// Work unit of the gate/up kernel: one tile (an expert and up to GEMV_MT of
// its tokens) x one group of 32 hidden units, i.e. 32 gate rows and the 32
// matching up rows: the 32 h values of a Q8_0 block are finished inside one
// block, so requantisation needs no second pass.  Warp w owns gate rows
// 4w..4w+3 and up rows 4w..4w+3 of the group; lane l owns 32-wide K blocks
// l, l+32, ...; each weight block is one 16-byte load.  The F32 accumulation
// of the per-block products follows one fixed order (blocks ascending, one
// fma each), so the hidden h, its Q8_0 codes and every later value come out
// the same bits as any other implementation of that order.
#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

// Stage the int8 activations of a tile's tokens into shared memory in split
// form (see block_dot), with each block's scale and the folded offset term
// MAGIC_I - 8*sum(q).
__device__ __forceinline__ void stage_tile(const int8_t *__restrict__ q, const float *__restrict__ d,
                                           int K, int m, const int32_t *__restrict__ rows_of,
                                           int row_limit, uint4 *xlo, uint4 *xhi, int *xcb,
                                           float *xd, int *status)
{
    const int NB = K / 32;
    for (int i = threadIdx.x; i < GEMV_MT * NB; i += blockDim.x) {
        const int t = i / NB, b = i - t * NB;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        int sum = 0;
        float dd = 0.0f;
        if (t < m) {
            const int row = rows_of[t];
            if (row >= 0 && row < row_limit) {
                const uint4 *src = reinterpret_cast<const uint4 *>(q + (size_t)row * K + (size_t)b * 32);
                split_block(src[0], src[1], &lo, &hi, &sum);
                dd = d[(size_t)row * NB + b];
            } else {
                set_status(status, ST_BAD_INDEX);
            }
        }
        xlo[i] = lo;
        xhi[i] = hi;
        xcb[i] = MAGIC_I - 8 * sum;
        xd[i] = dd;
    }
}

// Row dots of 8 rows x up to GEMV_MT tokens in the fixed F32 order
//     acc = 0; for b = 0, 1, ..., NB-1: acc = fma(d_b, (float)I_b, acc)
// (the per-row scale is applied by the caller).  The integer block dots are
// order-free, so lanes split K: lane l computes the blocks l, l+32, ... of
// all 8 rows.  After each chunk of 32 blocks the warp transposes its I values
// through shared memory (a 32 x 33 padded tile) so that lane c = r*GEMV_MT + t
// owns chain (row r, token t) and folds the chunk's 32 blocks in ascending
// order.  Returns lane c's chain value.
__device__ __forceinline__ float rows_x_tokens(const uint8_t *const (&rowp)[8], int NB, int m,
                                               const uint4 *xlo, const uint4 *xhi, const int *xcb,
                                               const float *xd, int (*ibuf)[33])
{
    const int lane = threadIdx.x & 31;
    const int t_own = lane % GEMV_MT;
    float acc = 0.0f;
    for (int j0 = 0; j0 < NB; j0 += 32) {
        const int b = j0 + lane;
        if (b < NB) {
            uint4 wv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) wv[r] = ld_stream(rowp[r] + (size_t)b * 16);
#pragma unroll
            for (int t = 0; t < GEMV_MT; ++t) {
                if (t < m) {
                    const uint4 lo = xlo[t * NB + b], hi = xhi[t * NB + b];
                    const int cb = xcb[t * NB + b];
#pragma unroll
                    for (int r = 0; r < 8; ++r) ibuf[r * GEMV_MT + t][lane] = block_dot(wv[r], lo, hi, cb);
                }
            }
        }
        __syncwarp();
        if (t_own < m) {
            const int nb = min(32, NB - j0);
            const float *dt = xd + t_own * NB + j0;
            const int *ib = ibuf[lane];
#pragma unroll 8
            for (int i = 0; i < nb; ++i) acc = __fmaf_rn(dt[i], __int_as_float(ib[i]) - MAGIC_F, acc);
        }
        __syncwarp();
    }
    return acc;
}

constexpr size_t IBUF_BYTES = 8 * 32 * 33 * sizeof(int);

size_t gateup_smem_bytes(int H)
{
    const int NB = H / 32;
    return (size_t)GEMV_MT * NB * (16 + 16 + 4 + 4) + (size_t)GEMV_MT * 64 * 4 + IBUF_BYTES;
}

size_t down_smem_bytes(int F)
{
    const int NB = F / 32;
    return (size_t)GEMV_MT * NB * (16 + 16 + 4 + 4) + IBUF_BYTES;
}

__global__ void __launch_bounds__(256, 2) k_gateup_gemv(ExpertArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int H = a.H, F = a.F, NB = H / 32, G = F / 32;
    uint4 *xlo = reinterpret_cast<uint4 *>(smem);
    uint4 *xhi = xlo + GEMV_MT * NB;
    int *xcb = reinterpret_cast<int *>(xhi + GEMV_MT * NB);
    float *xd = reinterpret_cast<float *>(xcb + GEMV_MT * NB);
    float *red = xd + GEMV_MT * NB;  // [GEMV_MT][64]: gate sums 0..31, up sums 32..63
    int(*ibuf)[33] = reinterpret_cast<int(*)[33]>(red + GEMV_MT * 64) + (threadIdx.x >> 5) * 32;
    __shared__ int s_tok[GEMV_MT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long units = (long)(*a.n_tiles) * G;

    for (long u = blockIdx.x; u < units; u += gridDim.x) {
        const int tile = (int)(u / G), g = (int)(u - (long)tile * G);
        const int e = a.tile_expert[tile], pos0 = a.tile_pos0[tile], m = a.tile_m[tile];
        const uint8_t *ew;
        const float *ers;
        if (e == a.E) {
            ew = a.shared_w4;
            ers = a.shared_rs;
        } else {
            ew = a.expert_w4 + (size_t)e * ((size_t)3 * F * H / 2);
            ers = a.expert_rs + (size_t)e * (2 * F + H);
        }
        if (threadIdx.x < GEMV_MT) s_tok[threadIdx.x] = (threadIdx.x < m) ? a.pos_token[pos0 + threadIdx.x] : 0;
        __syncthreads();
        stage_tile(a.qx, a.dx, H, m, s_tok, a.n_tok, xlo, xhi, xcb, xd, a.status);
        __syncthreads();

        const uint8_t *rowp[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = (r < 4) ? (32 * g + 4 * warp + r) : (F + 32 * g + 4 * warp + (r - 4));
            rowp[r] = ew + (size_t)row * (H / 2);
        }
        const float tot = rows_x_tokens(rowp, NB, m, xlo, xhi, xcb, xd, ibuf);
        {
            const int r = lane / GEMV_MT, t = lane % GEMV_MT;
            const int slot = (r < 4) ? (4 * warp + r) : (32 + 4 * warp + (r - 4));
            red[t * 64 + slot] = tot;
        }
        __syncthreads();
        if (warp < m) {
            const int t = warp, i = 32 * g + lane, pos = pos0 + t;
            const float gg = __fmul_rn(ers[i], red[t * 64 + lane]);
            const float uu = __fmul_rn(ers[F + i], red[t * 64 + 32 + lane]);
            const float h = __fmul_rn(__fmul_rn(gg, own_sigmoid(gg)), uu);
            float dq;
            const int q = q8_0_lane(h, &dq);
            a.qh[(size_t)pos * F + i] = (int8_t)q;
            if (lane == 0) a.dh[(size_t)pos * G + g] = dq;
            if (a.h_dbg) a.h_dbg[(size_t)pos * F + i] = h;
        }
        __syncthreads();
    }
}

// Down projection: one unit = one tile x 64 output rows (warp w: rows 8w..8w+7),
// K = F.  y[pos][row] = s_row * sum_b dh_b * I_b.
__global__ void __launch_bounds__(256, 2) k_down_gemv(ExpertArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int H = a.H, F = a.F, NB = F / 32, CH = H / 64;
    uint4 *xlo = reinterpret_cast<uint4 *>(smem);
    uint4 *xhi = xlo + GEMV_MT * NB;
    int *xcb = reinterpret_cast<int *>(xhi + GEMV_MT * NB);
    float *xd = reinterpret_cast<float *>(xcb + GEMV_MT * NB);
    int(*ibuf)[33] = reinterpret_cast<int(*)[33]>(xd + GEMV_MT * NB) + (threadIdx.x >> 5) * 32;
    __shared__ int s_rows[GEMV_MT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long units = (long)(*a.n_tiles) * CH;

    for (long u = blockIdx.x; u < units; u += gridDim.x) {
        const int tile = (int)(u / CH), c = (int)(u - (long)tile * CH);
        const int e = a.tile_expert[tile], pos0 = a.tile_pos0[tile], m = a.tile_m[tile];
        const uint8_t *ew;
        const float *ers;
        if (e == a.E) {
            ew = a.shared_w4;
            ers = a.shared_rs;
        } else {
            ew = a.expert_w4 + (size_t)e * ((size_t)3 * F * H / 2);
            ers = a.expert_rs + (size_t)e * (2 * F + H);
        }
        ew += (size_t)F * H;   // down matrix [H][F]
        ers += 2 * F;
        if (threadIdx.x < GEMV_MT) s_rows[threadIdx.x] = pos0 + threadIdx.x;
        __syncthreads();
        stage_tile(a.qh, a.dh, F, m, s_rows, a.P + a.n_tok, xlo, xhi, xcb, xd, a.status);
        __syncthreads();

        const uint8_t *rowp[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) rowp[r] = ew + (size_t)(64 * c + 8 * warp + r) * (F / 2);
        const float tot = rows_x_tokens(rowp, NB, m, xlo, xhi, xcb, xd, ibuf);
        const int r = lane / GEMV_MT, t = lane % GEMV_MT;
        if (t < m) {
            const int row = 64 * c + 8 * warp + r;
            a.y[(size_t)(pos0 + t) * H + row] = __fmul_rn(ers[row], tot);
        }
        __syncthreads();
    }
}

int max_gemv_tiles(int T, int k, int E)
{
    const long P = (long)T * k;
    const long routed = P / GEMV_MT + (P < E ? P : E) + 1;
    return (int)(routed + (T + GEMV_MT - 1) / GEMV_MT);
}

static unsigned gemv_grid(long units_ub, int num_sms)
{
    long cap = (long)num_sms * 8;
    long g = units_ub < cap ? units_ub : cap;
    return (unsigned)(g > 0 ? g : 1);
}

int launch_gateup_gemv(const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    static size_t configured = 0;
    const size_t smem = gateup_smem_bytes(a.H);
    if (smem > 48 * 1024 && smem != configured) {
        if (cudaFuncSetAttribute(k_gateup_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        configured = smem;
    }
    const long ub = (long)max_gemv_tiles(a.n_tok, a.k, a.E) * (a.F / 32);
    k_gateup_gemv<<<gemv_grid(ub, num_sms), 256, smem, st>>>(a);
    count_launch();
    return 0;
}

int launch_down_gemv(const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    const size_t smem = down_smem_bytes(a.F);
    static size_t configured = 0;
    if (smem > 48 * 1024 && smem != configured) {
        if (cudaFuncSetAttribute(k_down_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        configured = smem;
    }
    const long ub = (long)max_gemv_tiles(a.n_tok, a.k, a.E) * (a.H / 64);
    k_down_gemv<<<gemv_grid(ub, num_sms), 256, smem, st>>>(a);
    count_launch();
    return 0;
}

// out_t = y_shared,t + sum_r w_t,r * y_(pos of pair t*k+r), as an fma chain in
// rank order.  One thread per 4 outputs.
__global__ void __launch_bounds__(256) k_combine(const float *__restrict__ y, const int32_t *__restrict__ inv,
                                                 const float *__restrict__ w, int T, int k, int H, int P,
                                                 float *__restrict__ out)
{
    const int H4 = H / 4;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)T * H4) return;
    const int t = (int)(i / H4), j4 = (int)(i - (long)t * H4);
    const float4 *y4 = reinterpret_cast<const float4 *>(y);
    float4 acc = y4[(size_t)(P + t) * H4 + j4];
    for (int r = 0; r < k; ++r) {
        const int pos = inv[(size_t)t * k + r];
        if (pos < 0 || pos >= P) continue;
        const float wr = w[(size_t)t * k + r];
        const float4 v = y4[(size_t)pos * H4 + j4];
        acc.x = __fmaf_rn(wr, v.x, acc.x);
        acc.y = __fmaf_rn(wr, v.y, acc.y);
        acc.z = __fmaf_rn(wr, v.z, acc.z);
        acc.w = __fmaf_rn(wr, v.w, acc.w);
    }
    reinterpret_cast<float4 *>(out)[(size_t)t * H4 + j4] = acc;
}

int launch_combine(const float *y, const int32_t *inv, const float *w, int T, int k, int H, int P,
                   float *out, cudaStream_t st)
{
    const long n = (long)T * (H / 4);
    if (n == 0) return 0;
    k_combine<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, inv, w, T, k, H, P, out);
    count_launch();
    return 0;
}

// Stage-test helper: copy per-position rows into pair order (pair p reads
// position inv[p]; the shared rows P + t stay where they are).
__global__ void k_gather_pairs(const int32_t *__restrict__ inv, int T, int k, int P,
                               const int8_t *__restrict__ qh, const float *__restrict__ dh,
                               const float *__restrict__ y, int F, int H, int8_t *qh_out,
                               float *dh_out, float *y_out)
{
    const int p = blockIdx.x;
    if (p >= P + T) return;
    const int src = (p < P) ? inv[p] : p;
    if (src < 0 || src >= P + T) return;
    for (int i = threadIdx.x; i < F; i += blockDim.x) {
        if (qh_out) qh_out[(size_t)p * F + i] = qh[(size_t)src * F + i];
        if (dh_out && i < F / 32) dh_out[(size_t)p * (F / 32) + i] = dh[(size_t)src * (F / 32) + i];
    }
    if (y_out)
        for (int i = threadIdx.x; i < H; i += blockDim.x) y_out[(size_t)p * H + i] = y[(size_t)src * H + i];
}

int launch_gather_pairs(const int32_t *inv, int T, int k, int P, const int8_t *qh, const float *dh,
                        const float *y, int F, int H, int8_t *qh_out, float *dh_out, float *y_out,
                        cudaStream_t st)
{
    if (P + T == 0) return 0;
    k_gather_pairs<<<P + T, 256, 0, st>>>(inv, T, k, P, qh, dh, y, F, H, qh_out, dh_out, y_out);
    count_launch();
    return 0;
}

}  // namespace coli
