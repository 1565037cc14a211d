// k_route.cu -- F32 sigmoid router (logits, top-k, renormalisation) and the
// batch-union dispatch (stable counting sort of token->expert pairs).
//
// Router: DeepSeek-V3-style sigmoid gating with a selection-only bias and a
// shared expert ("Open-source engine that ran 744B GLM-5.2 on a 25GB-RAM
// laptop", jeff.news, section "Attention and kernels"), kept in F32
// ("GLM-5.2-colibri-int4" model card, section "Good to know").
// Dispatch: prefill routes the union of the batch's experts in one pass
// ("Colibri: an AI engine running a 744B model in 25GB of RAM", alphamatch.ai,
// section "Technical excellence").
#include <climits>

#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

// ---------------------------------------------------------------------------
// Router logits in one fixed F32 order, so that expert choices are bit-exact
// wherever they are computed.  The H inputs form chunks of 4 consecutive
// elements; chunk c accumulates into partial p[c mod 256] (thread c mod 256 of
// the block), chunks ascending, elements of a chunk ascending, each step an
// fma from p = +0.  The 256 partials fold as 8 groups of 32 by an xor
// butterfly (p[j] + p[j ^ o], o = 16..1: a warp shuffle), and the 8 group sums
// fold the same way with o = 4, 2, 1.
// A block computes ET experts x TT tokens; each weight and input chunk is
// loaded once per block.
// ---------------------------------------------------------------------------
template <int ET, int TT>
__global__ void __launch_bounds__(256) k_router_logits(const float *__restrict__ x, int T, int H,
                                                       const float *__restrict__ W, int E,
                                                       float *__restrict__ logits)
{
    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const int e0 = blockIdx.x * ET, t0 = blockIdx.y * TT;
    float acc[ET][TT];
#pragma unroll
    for (int e = 0; e < ET; ++e)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[e][t] = 0.0f;

    const int nch = H >> 2;
    for (int c = j; c < nch; c += 256) {
        float4 wv[ET], xv[TT];
#pragma unroll
        for (int e = 0; e < ET; ++e)
            wv[e] = (e0 + e < E) ? __ldg(reinterpret_cast<const float4 *>(W + (size_t)(e0 + e) * H) + c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < TT; ++t)
            xv[t] = (t0 + t < T) ? __ldg(reinterpret_cast<const float4 *>(x + (size_t)(t0 + t) * H) + c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < ET; ++e)
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float p = acc[e][t];
                p = __fmaf_rn(xv[t].x, wv[e].x, p);
                p = __fmaf_rn(xv[t].y, wv[e].y, p);
                p = __fmaf_rn(xv[t].z, wv[e].z, p);
                p = __fmaf_rn(xv[t].w, wv[e].w, p);
                acc[e][t] = p;
            }
    }

    __shared__ float red[ET * TT][8];
#pragma unroll
    for (int e = 0; e < ET; ++e)
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float v = acc[e][t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, o));
            if (lane == 0) red[e * TT + t][warp] = v;
        }
    __syncthreads();
    for (int i = j; i < ET * TT; i += 256) {
        float s[8], tmp[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) s[w] = red[i][w];
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
#pragma unroll
            for (int w = 0; w < 8; ++w) tmp[w] = __fadd_rn(s[w], s[w ^ o]);
#pragma unroll
            for (int w = 0; w < 8; ++w) s[w] = tmp[w];
        }
        int e = e0 + i / TT, t = t0 + i % TT;
        if (e < E && t < T) logits[(size_t)t * E + e] = s[0];
    }
}

int launch_router_logits(const float *x, int T, int H, const float *W, int E, float *logits,
                         cudaStream_t st)
{
    if (T <= 0) return 0;
    if (T == 1) {
        k_router_logits<1, 1><<<dim3(E, 1), 256, 0, st>>>(x, T, H, W, E, logits);
    } else if (T <= 4) {
        k_router_logits<1, 4><<<dim3(E, 1), 256, 0, st>>>(x, T, H, W, E, logits);
    } else {
        k_router_logits<8, 8><<<dim3((E + 7) / 8, (T + 7) / 8), 256, 0, st>>>(x, T, H, W, E, logits);
    }
    count_launch();
    return 0;
}

// ---------------------------------------------------------------------------
// Top-k with lowest-index ties, one warp per token (E <= 256: 8 experts per
// lane).  sigma_e = sigmoid(logit_e); key_e = sigma_e + bias_e (selection
// only); S = sum of the chosen sigma in rank order from 0;
// w_r = (sigma_r / S) * routed_scale.
// ---------------------------------------------------------------------------
constexpr int MAX_K = 16;

// Top-k of one token's logits by one warp.  Lane 0 writes the experts in rank
// order to idx_out[0..k) and their sigma to sig_out[0..k); every lane returns
// S = the sum of the chosen sigma in rank order.  The rounds are a rolled
// loop: this runs once per token at the end of routing, where a compact body
// matters more than unrolling.
__device__ __noinline__ float warp_topk(const float *logits_row, int E, int k,
                                        const float *__restrict__ bias, int *idx_out, float *sig_out)
{
    const int lane = threadIdx.x & 31;
    float sig[8], key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int e = lane + 32 * i;
        if (e < E) {
            sig[i] = own_sigmoid(__ldcg(logits_row + e));
            key[i] = __fadd_rn(sig[i], bias[e]);
        } else {
            sig[i] = 0.0f;
            key[i] = -__int_as_float(0x7f800000);
        }
    }
    unsigned taken = 0;
    float S = 0.0f;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        float bv = -__int_as_float(0x7f800000);
        int be = INT_MAX;
        float bs = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (key[i] > bv || be == INT_MAX)) {
                bv = key[i];
                be = e;
                bs = sig[i];
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            float ov = __shfl_xor_sync(FULL, bv, o);
            int oe = __shfl_xor_sync(FULL, be, o);
            float os = __shfl_xor_sync(FULL, bs, o);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
                bs = os;
            }
        }
        if (be != INT_MAX && (be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) {
            idx_out[r] = (be == INT_MAX) ? -1 : be;
            sig_out[r] = bs;
        }
        S = __fadd_rn(S, bs);
    }
    return S;
}

__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits, int T, int E, int k,
                                              const float *__restrict__ bias, float scale,
                                              int32_t *__restrict__ idx, float *__restrict__ w)
{
    __shared__ int s_idx[8][MAX_K];
    __shared__ float s_sig[8][MAX_K];
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (t >= T) return;
    const float S = warp_topk(logits + (size_t)t * E, E, k, bias, s_idx[warp], s_sig[warp]);
    __syncwarp();
    if (lane < k) {
        idx[(size_t)t * k + lane] = s_idx[warp][lane];
        w[(size_t)t * k + lane] = __fmul_rn(__fdiv_rn(s_sig[warp][lane], S), scale);
    }
}

int launch_topk(const float *logits, int T, int E, int k, const float *bias, float routed_scale,
                int32_t *idx, float *w, cudaStream_t st)
{
    if (T <= 0) return 0;
    unsigned grid = (unsigned)(((long)T * 32 + 255) / 256);
    k_topk<<<grid, 256, 0, st>>>(logits, T, E, k, bias, routed_scale, idx, w);
    count_launch();
    return 0;
}

// ---------------------------------------------------------------------------
// Dispatch: one block of 1024 threads.  Pair p = t*k + r goes to position
// offsets[e_p] + #{p' < p : e_p' = e_p} (a stable counting sort, so the
// tokens of an expert stay in ascending order).  Pairs are ranked 1024 at a
// time: warp-level match gives the rank inside a warp, a per-(warp, expert)
// count table scanned across the 32 warps gives the rank inside the chunk,
// and a running base per expert carries it across chunks.  All integer, no
// order-dependent atomics.
// Also emits pos_token (token of each position; the shared expert's rows sit
// at P + t) and the GEMV tile list: shared expert tiles first, then each
// routed expert's tokens in tiles of GEMV_MT, experts ascending.
// ---------------------------------------------------------------------------
constexpr int DISPATCH_THREADS = 1024;
constexpr int MAX_E = 256;

// Warp 0: exclusive scans of the per-expert counts and tile counts (E <= 256,
// 8 per lane).  Writes counts/offsets (global), s_base/s_tile0 (shared) and
// the total tile count (shared experts' tiles first).
__device__ __noinline__ void scan_experts(const int *s_cnt, int E, int T, int32_t *counts,
                                          int32_t *offsets, int *s_base, int *s_tile0,
                                          int *s_ntiles)
{
    // rolled loops: runs once per forward on code no other warp has fetched
    const int lane = threadIdx.x & 31;
    int sum = 0, tsum = 0;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        const int v = (e < E) ? s_cnt[e] : 0;
        sum += v;
        tsum += (v + GEMV_MT - 1) / GEMV_MT;
    }
    int inc = sum, tinc = tsum;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
        int a = __shfl_up_sync(FULL, inc, o);
        int b = __shfl_up_sync(FULL, tinc, o);
        if (lane >= o) { inc += a; tinc += b; }
    }
    int run = inc - sum, trun = tinc - tsum;
    const int shared_tiles = (T + GEMV_MT - 1) / GEMV_MT;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        const int v = (e < E) ? s_cnt[e] : 0;
        if (e < E) {
            s_base[e] = run;
            offsets[e] = run;
            counts[e] = v;
            s_tile0[e] = shared_tiles + trun;
        }
        run += v;
        trun += (v + GEMV_MT - 1) / GEMV_MT;
    }
    if (lane == 31) {
        offsets[E] = inc;
        *s_ntiles = shared_tiles + tinc;
    }
}

// All threads of the block: the tile list (shared expert's tiles, then each
// routed expert's tokens in tiles of GEMV_MT) and pos_token of the shared rows.
__device__ __forceinline__ void write_tiles(int T, int P, int E, const int *s_cnt, const int *s_tile0,
                                            const int32_t *offsets_sh, int s_ntiles,
                                            int32_t *pos_token, int32_t *tile_expert,
                                            int32_t *tile_pos0, int32_t *tile_m, int32_t *n_tiles)
{
    const int tid = threadIdx.x;
    for (int t = tid; t < T; t += blockDim.x) pos_token[P + t] = t;
    const int shared_tiles = (T + GEMV_MT - 1) / GEMV_MT;
    for (int j = tid; j < shared_tiles; j += blockDim.x) {
        tile_expert[j] = E;
        tile_pos0[j] = P + j * GEMV_MT;
        tile_m[j] = min(GEMV_MT, T - j * GEMV_MT);
    }
    for (int e = tid; e < E; e += blockDim.x) {
        const int cnt = s_cnt[e], t0 = s_tile0[e], off = offsets_sh[e];
        for (int j = 0; j * GEMV_MT < cnt; ++j) {
            tile_expert[t0 + j] = e;
            tile_pos0[t0 + j] = off + j * GEMV_MT;
            tile_m[t0 + j] = min(GEMV_MT, cnt - j * GEMV_MT);
        }
    }
    if (tid == 0) *n_tiles = s_ntiles;
}

// ---------------------------------------------------------------------------
// Dispatch: one block of 1024 threads.  Pair p = t*k + r goes to position
// offsets[e_p] + #{p' < p : e_p' = e_p} (a stable counting sort, so the
// tokens of an expert stay in ascending order).  Pairs are ranked 1024 at a
// time: warp-level match gives the rank inside a warp, a per-(warp, expert)
// count table scanned across the 32 warps gives the rank inside the chunk,
// and a running base per expert carries it across chunks.  All integer, no
// order-dependent atomics.  Also emits pos_token, the tile list, and zeroes
// the expert kernel's counters.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(DISPATCH_THREADS) k_dispatch(
    const int32_t *__restrict__ idx, int T, int k, int E, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
    int32_t *__restrict__ pos_token, int32_t *__restrict__ tile_expert,
    int32_t *__restrict__ tile_pos0, int32_t *__restrict__ tile_m, int32_t *__restrict__ n_tiles,
    int *sync, int n_sync, int *status)
{
    __shared__ int s_cnt[MAX_E];
    __shared__ int s_base[MAX_E];
    __shared__ int s_off[MAX_E];
    __shared__ int s_wc[32][MAX_E];
    __shared__ int s_tile0[MAX_E];
    __shared__ int s_ntiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = T * k;

    for (int i = tid; i < n_sync; i += DISPATCH_THREADS) sync[i] = 0;
    if (tid < MAX_E) s_cnt[tid] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += DISPATCH_THREADS) {
        int e = idx[p];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
        else set_status(status, ST_BAD_INDEX);
    }
    __syncthreads();
    if (warp == 0) scan_experts(s_cnt, E, T, counts, offsets, s_base, s_tile0, &s_ntiles);
    __syncthreads();
    if (tid < E) s_off[tid] = s_base[tid];

    for (int c0 = 0; c0 < P; c0 += DISPATCH_THREADS) {
        for (int i = tid; i < 32 * MAX_E; i += DISPATCH_THREADS) (&s_wc[0][0])[i] = 0;
        __syncthreads();
        const int p = c0 + tid;
        int e = (p < P) ? idx[p] : -1;
        const bool valid = (e >= 0 && e < E);
        if (!valid) e = -1;
        const unsigned peers = __match_any_sync(FULL, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (valid && rank == 0) s_wc[warp][e] = __popc(peers);
        __syncthreads();
        int chunk_total = 0;
        if (tid < E) {
            for (int w = 0; w < 32; ++w) {
                int c = s_wc[w][tid];
                s_wc[w][tid] = chunk_total;
                chunk_total += c;
            }
        }
        __syncthreads();
        if (valid) {
            int pos = s_base[e] + s_wc[warp][e] + rank;
            perm[pos] = p;
            inv[p] = pos;
            pos_token[pos] = p / k;
        } else if (p < P) {
            inv[p] = -1;
        }
        __syncthreads();
        if (tid < E) s_base[tid] += chunk_total;
        __syncthreads();
    }
    write_tiles(T, P, E, s_cnt, s_tile0, s_off, s_ntiles, pos_token, tile_expert, tile_pos0,
                tile_m, n_tiles);
}

int launch_dispatch(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv, int32_t *pos_token, int32_t *tile_expert,
                    int32_t *tile_pos0, int32_t *tile_m, int32_t *n_tiles, int *sync, int n_sync,
                    int *status, cudaStream_t st)
{
    k_dispatch<<<1, DISPATCH_THREADS, 0, st>>>(idx, T, k, E, counts, offsets, perm, inv, pos_token,
                                               tile_expert, tile_pos0, tile_m, n_tiles, sync, n_sync,
                                               status);
    count_launch();
    return 0;
}

// Order-preserving 64-bit image of a (selection key, expert) pair: a larger
// key first, then the lower expert index (the selection order of the
// sigmoid router); 0 lies below the image of every finite key.  Keys are
// sigma + bias, finite; adding +0 maps -0 to +0 so that equal keys have
// equal images.
__device__ __forceinline__ unsigned long long route_image(float key, int e)
{
    const uint32_t u = __float_as_uint(__fadd_rn(key, 0.0f));
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}

// Bitonic sort of one value per lane across the warp, largest in lane 0.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long c, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long o = __shfl_xor_sync(FULL, c, stride);
            // the lower lane of a pair keeps the larger value in blocks that
            // end up descending (all of them at the last size)
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            c = keep_max ? (c > o ? c : o) : (c < o ? c : o);
        }
    }
    return c;
}

// ---------------------------------------------------------------------------
// Small batches (T <= ROUTE_SMALL_MAX_T) route in a single launch of E blocks:
// every block quantises a share of x and computes the logits of its expert
// for all T tokens (same fixed order as k_router_logits); the last block to
// finish (a completion counter) runs top-k, the stable dispatch of the
// T*k <= 128 pairs, the tile list, and zeroes the expert kernel's counters.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) k_route_small(const RouteArgs ra)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = ra.T, H = ra.H, E = ra.E, k = ra.k;
    const int e = blockIdx.x;
    // the expert kernel may start launching now; it waits for this grid's
    // results (griddepcontrol.wait) before reading any of them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // 1. Q8_0 of x: warps of all blocks share the T*H/32 blocks
    const long nblk = (long)T * H / 32;
    for (long blk = (long)blockIdx.x * 8 + warp; blk < nblk; blk += (long)gridDim.x * 8) {
        float d;
        const int qv = q8_0_lane(ra.x[blk * 32 + lane], &d);
        ra.qx[blk * 32 + lane] = (int8_t)qv;
        if (lane == 0) ra.dx[blk] = d;
    }

    // 2. logits of expert e for every token (each thread's weight chunks are
    //    loaded together, LG at a time, so the row costs one or two round trips)
    float acc[ROUTE_SMALL_MAX_T];
#pragma unroll
    for (int t = 0; t < ROUTE_SMALL_MAX_T; ++t) acc[t] = 0.0f;
    const float4 *w4 = reinterpret_cast<const float4 *>(ra.W + (size_t)e * H);
    constexpr int LG = 8;
    for (int c0 = tid; c0 < H / 4; c0 += 256 * LG) {
        float4 wv[LG];
#pragma unroll
        for (int u = 0; u < LG; ++u) {
            const int c = c0 + 256 * u;
            wv[u] = (c < H / 4) ? __ldg(w4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int t = 0; t < ROUTE_SMALL_MAX_T; ++t) {
            if (t < T) {
                const float4 *x4 = reinterpret_cast<const float4 *>(ra.x + (size_t)t * H);
                float4 xv[LG];
#pragma unroll
                for (int u = 0; u < LG; ++u) {
                    const int c = c0 + 256 * u;
                    xv[u] = (c < H / 4) ? __ldg(x4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float p = acc[t];
#pragma unroll
                for (int u = 0; u < LG; ++u) {
                    if (c0 + 256 * u < H / 4) {      // chunks ascending, elements ascending
                        p = __fmaf_rn(xv[u].x, wv[u].x, p);
                        p = __fmaf_rn(xv[u].y, wv[u].y, p);
                        p = __fmaf_rn(xv[u].z, wv[u].z, p);
                        p = __fmaf_rn(xv[u].w, wv[u].w, p);
                    }
                }
                acc[t] = p;
            }
        }
    }
    __shared__ float red[ROUTE_SMALL_MAX_T][8];
#pragma unroll
    for (int t = 0; t < ROUTE_SMALL_MAX_T; ++t) {
        if (t < T) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, o));
            if (lane == 0) red[t][warp] = v;
        }
    }
    __syncthreads();
    if (tid < T) {
        float s8[8], tmp[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) s8[w] = red[tid][w];
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
#pragma unroll
            for (int w = 0; w < 8; ++w) tmp[w] = __fadd_rn(s8[w], s8[w ^ o]);
#pragma unroll
            for (int w = 0; w < 8; ++w) s8[w] = tmp[w];
        }
        ra.logits[(size_t)tid * E + e] = s8[0];
        // sigma and the selection key here, in every block, rather than in
        // the last block's serial tail
        const float sg = own_sigmoid(s8[0]);
        ra.sig[(size_t)tid * E + e] = sg;
        ra.key[(size_t)tid * E + e] = __fadd_rn(sg, __ldg(ra.bias + e));
    }

    // 3. the last block routes
    __shared__ int s_last;
    unsigned long long *tr = ra.trace;
    auto stamp = [&](int i) {
        if (tr && tid == 0) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
            tr[i] = t;
        }
    };
    stamp(0 + 16 * (blockIdx.x == 0));
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(ra.route_counter, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    stamp(1);
    __threadfence();
    if (tid == 0) *ra.route_counter = 0;

    __shared__ int s_idx[ROUTE_SMALL_MAX_T * MAX_K];
    __shared__ float s_sig[ROUTE_SMALL_MAX_T * MAX_K];
    __shared__ int s_cnt[MAX_E], s_base[MAX_E], s_tile0[MAX_E], s_off[MAX_E];
    __shared__ int s_ntiles;
    __shared__ float s_key[ROUTE_SMALL_MAX_T][MAX_E], s_sg[ROUTE_SMALL_MAX_T][MAX_E];
    if (T == 1) {
        // ---- one token: the k best of E <= 256 keys, then dispatch of k
        //      distinct experts, in three barrier-separated phases ----
        __shared__ unsigned long long s_cand[8 * MAX_K];
        // (a) each warp sorts the images of its 32 experts and offers its k best
        unsigned long long c = 0;
        if (tid < E) {
            s_sg[0][tid] = __ldcg(ra.sig + tid);
            c = route_image(__ldcg(ra.key + tid), tid);
        }
        c = warp_sort_desc(c, lane);
        if (lane < k) s_cand[warp * k + lane] = c;
        __syncthreads();
        stamp(7);
        // (b) the rank of each candidate among the 8k (images are distinct
        //     for valid experts; the k best are valid since E >= k)
        const int nc = 8 * k;
        if (tid < nc) {
            const unsigned long long ci = s_cand[tid];
            int rank = 0;
#pragma unroll 8
            for (int j = 0; j < nc; ++j) rank += (s_cand[j] > ci);
            if (rank < k) {
                const int sel = ci ? (int)(0xFFFFFFFFu - (uint32_t)ci) : -1;
                s_idx[rank] = sel;
                s_sig[rank] = sel >= 0 ? s_sg[0][sel] : 0.0f;
            }
        }
        __syncthreads();
        stamp(8);
        // (c) weights, positions and tiles of the k pairs (warp 0), counts and
        //     offsets of every expert (all threads).  Position of a pair = the
        //     number of chosen experts with a lower index; tile 0 is the
        //     shared expert's, tile 1 + pos the pair's.
        if (warp == 0) {
            const bool act = lane < k;
            const int e_r = act ? s_idx[lane] : 0;
            const float sg_r = act ? s_sig[lane] : 0.0f;
            float S = 0.0f;
            int pos = 0;
#pragma unroll 1
            for (int r = 0; r < k; ++r) {
                S = __fadd_rn(S, __shfl_sync(FULL, sg_r, r));
                pos += (__shfl_sync(FULL, e_r, r) < e_r);
            }
            if (act) {
                ra.idx[lane] = e_r;
                ra.wts[lane] = __fmul_rn(__fdiv_rn(sg_r, S), ra.routed_scale);
                if (e_r >= 0 && e_r < E) {
                    ra.perm[pos] = lane;
                    ra.inv[lane] = pos;
                    ra.pos_token[pos] = 0;
                    ra.tile_expert[1 + pos] = e_r;
                    ra.tile_pos0[1 + pos] = pos;
                    ra.tile_m[1 + pos] = 1;
                } else {
                    ra.inv[lane] = -1;
                    set_status(ra.status, ST_BAD_INDEX);
                }
            }
            if (lane == 0) {
                ra.pos_token[k] = 0;
                ra.tile_expert[0] = E;
                ra.tile_pos0[0] = k;
                ra.tile_m[0] = 1;
                *ra.n_tiles = 1 + k;
                ra.offsets[E] = k;
            }
        }
        for (int e2 = tid; e2 < E; e2 += 256) {
            int below = 0, hit = 0;
#pragma unroll 1
            for (int r = 0; r < k; ++r) {
                const int er = s_idx[r];
                below += (er < e2);
                hit += (er == e2);
            }
            ra.counts[e2] = hit;
            ra.offsets[e2] = below;
        }
        __syncthreads();
        stamp(2);
        stamp(3);
        stamp(4);
        stamp(5);
        stamp(6);
        return;
    }
    // sigma and selection key of every (token, expert), computed by the
    // expert's block
#pragma unroll 1
    for (int i = tid; i < T * E; i += 256) {
        const int t = i / E, ee = i - t * E;
        s_sg[t][ee] = __ldcg(ra.sig + (size_t)t * E + ee);
        s_key[t][ee] = __ldcg(ra.key + (size_t)t * E + ee);
    }
    __syncthreads();
    stamp(7);
    if (warp < T) {
        // Several tokens: one warp per token, k rounds of a warp-wide argmax
        // over the experts not yet taken under the selection order: larger
        // key first, then lower index.
        // Lane l holds experts l, l+32, ...
        const int t = warp;
        unsigned taken = 0;                       // bit i: expert lane + 32 i taken
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            float bk = 0.0f;
            int be = -1;
#pragma unroll 1
            for (int i = 0; i < MAX_E / 32; ++i) {
                const int ee = lane + 32 * i;
                if (ee < E && !((taken >> i) & 1u)) {
                    const float kv = s_key[t][ee];
                    if (be < 0 || kv > bk) {      // ascending ee: the first of equal keys stays
                        bk = kv;
                        be = ee;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ok = __shfl_xor_sync(FULL, bk, o);
                const int oe = __shfl_xor_sync(FULL, be, o);
                if (oe >= 0 && (be < 0 || ok > bk || (ok == bk && oe < be))) {
                    bk = ok;
                    be = oe;
                }
            }
            if (be >= 0 && (be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == 0) {
                s_idx[t * k + r] = be;
                s_sig[t * k + r] = be >= 0 ? s_sg[t][be] : 0.0f;
            }
        }
    }
    __syncthreads();
    stamp(8);
    // S = sum of the chosen sigma in rank order (one thread per token), then
    // the weights, one pair per thread
    __shared__ float s_S[ROUTE_SMALL_MAX_T];
    if (tid < T) {
        float S = 0.0f;
#pragma unroll 1
        for (int r = 0; r < k; ++r) S = __fadd_rn(S, s_sig[tid * k + r]);
        s_S[tid] = S;
    }
    __syncthreads();
    if (tid < T * k) {
        ra.idx[tid] = s_idx[tid];
        ra.wts[tid] = __fmul_rn(__fdiv_rn(s_sig[tid], s_S[tid / k]), ra.routed_scale);
    }
    __syncthreads();
    stamp(2);
    const int P = T * k;
    for (int ee = tid; ee < MAX_E; ee += 256) {
        int c = 0;
        for (int p = 0; p < P; ++p) c += (s_idx[p] == ee);
        s_cnt[ee] = (ee < E) ? c : 0;
    }
    if (tid < P && (s_idx[tid] < 0 || s_idx[tid] >= E)) set_status(ra.status, ST_BAD_INDEX);
    __syncthreads();
    stamp(3);
    {
        // exclusive scans of the counts and tile counts: one expert per thread,
        // warp scans plus a scan of the eight warp totals
        __shared__ int s_wsum[8], s_wtsum[8];
        const int v = (tid < E) ? s_cnt[tid] : 0;
        const int nt = (v + GEMV_MT - 1) / GEMV_MT;
        int inc = v, tinc = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(FULL, inc, o), b = __shfl_up_sync(FULL, tinc, o);
            if (lane >= o) { inc += a; tinc += b; }
        }
        if (lane == 31) { s_wsum[warp] = inc; s_wtsum[warp] = tinc; }
        __syncthreads();
        int base = 0, tbase = 0;
        for (int w2 = 0; w2 < warp; ++w2) { base += s_wsum[w2]; tbase += s_wtsum[w2]; }
        const int shared_tiles = (T + GEMV_MT - 1) / GEMV_MT;
        if (tid < E) {
            s_base[tid] = base + inc - v;
            ra.offsets[tid] = base + inc - v;
            ra.counts[tid] = v;
            s_tile0[tid] = shared_tiles + tbase + tinc - nt;
        }
        if (tid == 255) {
            ra.offsets[E] = base + inc;
            s_ntiles = shared_tiles + tbase + tinc;
        }
    }
    __syncthreads();
    if (tid < E) s_off[tid] = s_base[tid];
    __syncthreads();
    stamp(4);
    if (tid < P) {
        const int ee = s_idx[tid];
        if (ee >= 0 && ee < E) {
            int rank = 0;
            for (int p = 0; p < tid; ++p) rank += (s_idx[p] == ee);
            const int pos = s_off[ee] + rank;
            ra.perm[pos] = tid;
            ra.inv[tid] = pos;
            ra.pos_token[pos] = tid / k;
        } else {
            ra.inv[tid] = -1;
        }
    }
    stamp(5);
    write_tiles(T, P, E, s_cnt, s_tile0, s_off, s_ntiles, ra.pos_token, ra.tile_expert,
                ra.tile_pos0, ra.tile_m, ra.n_tiles);
    __syncthreads();
    stamp(6);
}

int launch_route_small(const RouteArgs &r, cudaStream_t st)
{
    k_route_small<<<r.E, 256, 0, st>>>(r);
    count_launch();
    return 0;
}

// Tile list for a single expert (index 0) over positions 0..n-1.
__global__ void k_single_expert_tiles(int n, int32_t *pos_token, int32_t *tile_expert,
                                      int32_t *tile_pos0, int32_t *tile_m, int32_t *n_tiles,
                                      int *sync, int n_sync)
{
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) pos_token[i] = i;
    int nt = (n + GEMV_MT - 1) / GEMV_MT;
    if (i < nt) {
        tile_expert[i] = 0;
        tile_pos0[i] = i * GEMV_MT;
        tile_m[i] = min(GEMV_MT, n - i * GEMV_MT);
    }
    for (int j = i; j < n_sync; j += gridDim.x * blockDim.x) sync[j] = 0;
    if (i == 0) *n_tiles = nt;
}

int launch_single_expert_tiles(int n, int32_t *pos_token, int32_t *tile_expert, int32_t *tile_pos0,
                               int32_t *tile_m, int32_t *n_tiles, int *sync, int n_sync,
                               cudaStream_t st)
{
    k_single_expert_tiles<<<(n + 255) / 256, 256, 0, st>>>(n, pos_token, tile_expert, tile_pos0,
                                                          tile_m, n_tiles, sync, n_sync);
    count_launch();
    return 0;
}

}  // namespace coli
