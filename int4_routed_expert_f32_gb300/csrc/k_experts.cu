// k_experts.cu -- persistent expert kernel: gate/up with SiLU*up and Q8_0
// requantisation of h, down, and the gate-weighted combine, in one launch.
//
// Method (int4 weights x Q8_0 int8 activations, int32 per 32-block, then F32
// scaling; SwiGLU experts plus a shared expert): "colibri: a pure-C inference
// engine ..." (discuss.pytorch.kr), section "Key features"; "Open-source engine
// that ran 744B GLM-5.2 on a 25GB-RAM laptop" (jeff.news), section "Attention
// and kernels"; "Colibri: an AI engine running a 744B model in 25GB of RAM"
// (alphamatch.ai), section "Optimised integer kernels".
//
// Structure (one CTA per SM, 8 consumer warps + 1 producer warp):
//   * Work units: every gate/up unit (a tile of <= GEMV_MT tokens of one
//     expert x 32 hidden units = 32 gate rows + 32 up rows), then every down
//     unit (a tile x 64 output rows).  Each block takes a contiguous share of
//     the gate/up units and then of the down units (a static schedule known to
//     producer and consumers alike).
//   * The producer streams each unit's weights through a ring of NSTAGE
//     shared-memory stages with 3-D TMA tile loads.  A stage holds 64 weight
//     rows x NSUB sub-chunks of 128 bytes (256 weights) each; a sub-chunk is
//     one swizzled TMA box (128-byte swizzle), L2 evict-first.  Each stage
//     completes on its mbarrier; consumers release it through a second one.
//   * Consumers: a quad of lanes per weight row, lane q of the quad owns
//     sub-chunk q (8 blocks of 32 weights); dp4a block dots.  The F32
//     accumulation of the row runs in block order (acc = fma(d_b, I_b, acc),
//     b ascending): lane 0 folds its 8 blocks, hands acc to lane 1, and so on.
//   * A down unit needs the h codes of its whole tile: it waits (bounded) on
//     the tile's gate/up completion counter.  Each 64-row output chunk is
//     combined by the block that ran the chunk's down unit of the last tile,
//     after (bounded) waiting for the chunk's down units of the other tiles.
// Counters are zeroed by the dispatch step that precedes the launch.
#include <cuda.h>

#include "coli_common.cuh"
#include "coli_internal.h"
#include "tma.cuh"

namespace coli {

constexpr int NSTAGE = 4;
constexpr int STAGE_ROWS = 64;
constexpr int KC_MAX = 128;
constexpr int NSUB_MAX = 4;
constexpr int SUB_BYTES = STAGE_ROWS * KC_MAX;      // 8 KB: one sub-chunk of 64 rows
constexpr int STAGE_BYTES = NSUB_MAX * SUB_BYTES;   // 32 KB
constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int EXPERT_THREADS = CONSUMERS + 32;
constexpr int BAR_CONSUMERS = 1;                   // named barrier id (0 = __syncthreads)
constexpr uint64_t WAIT_NS = 2000000000ull;        // 2 s bound on every wait

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > WAIT_NS) return false;
    }
}

struct ExpertSmem {
    int abort;
    int tok[GEMV_MT];
    alignas(8) uint64_t full[NSTAGE];
    alignas(8) uint64_t empty[NSTAGE];
};

size_t experts_smem_bytes(int H, int F)
{
    const int NB = (H > F ? H : F) / 32;
    size_t act = (size_t)GEMV_MT * NB * (16 + 16 + 4 + 4);
    size_t red = (size_t)GEMV_MT * 64 * 4;
    return 1024 /*align slack*/ + (size_t)NSTAGE * STAGE_BYTES + act + red + sizeof(ExpertSmem);
}

// Split-form activations of one tile into shared memory (see block_dot).
__device__ __forceinline__ void stage_acts(const int8_t *__restrict__ q, const float *__restrict__ d,
                                           int K, int m, const int *rows, int row_limit,
                                           uint4 *xlo, uint4 *xhi, int *xcb, float *xd, int *status)
{
    const int NB = K / 32;
    for (int i = threadIdx.x; i < GEMV_MT * NB; i += CONSUMERS) {
        const int t = i / NB, b = i - t * NB;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        int sum = 0;
        float dd = 0.0f;
        if (t < m) {
            const int row = rows[t];
            if (row >= 0 && row < row_limit) {
                const uint4 *src = reinterpret_cast<const uint4 *>(q + (size_t)row * K + (size_t)b * 32);
                split_block(__ldcg(src), __ldcg(src + 1), &lo, &hi, &sum);
                dd = __ldcg(d + (size_t)row * NB + b);
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

// Integer dot of a block with the low and high nibbles accumulated apart:
// the high nibbles are used in place (16 x nibble), so no shifts are needed.
__device__ __forceinline__ int block_dot_i(uint4 w, uint4 lo, uint4 hi, int cb)
{
    int a = cb, h = 0;
    a = dp4a_us(w.x & 0x0F0F0F0Fu, (int)lo.x, a);
    h = dp4a_us(w.x & 0xF0F0F0F0u, (int)hi.x, h);
    a = dp4a_us(w.y & 0x0F0F0F0Fu, (int)lo.y, a);
    h = dp4a_us(w.y & 0xF0F0F0F0u, (int)hi.y, h);
    a = dp4a_us(w.z & 0x0F0F0F0Fu, (int)lo.z, a);
    h = dp4a_us(w.z & 0xF0F0F0F0u, (int)hi.z, h);
    a = dp4a_us(w.w & 0x0F0F0F0Fu, (int)lo.w, a);
    h = dp4a_us(w.w & 0xF0F0F0F0u, (int)hi.w, h);
    return a + (h >> 4);     // = sum(nibble * x) - 8 * sum(x), exactly
}

// Integer block dots of one pipeline stage for this lane (row r, sub-chunk q):
// dst[t][jj] = MAGIC_I + I(block b0 + (jj + rot) mod BPS, token t).  Waits for
// the stage, and releases it once the dots are done.  False if the wait gave up.
template <int MT>
__device__ __forceinline__ bool stage_dots(uint64_t *full, uint64_t *empty, const unsigned char *ring,
                                           long &it, const int (&woff)[8], const uint4 *xlo,
                                           const uint4 *xhi, const int *xcb, int sub, int BPS, int rot,
                                           int NB, int m, bool active, int lane, int (&dst)[MT][8])
{
    const int slot = (int)(it % NSTAGE);
    const uint32_t round = (uint32_t)(it / NSTAGE);
    if (!mbar_wait_bounded(&full[slot], round & 1)) return false;
    const unsigned char *base = ring + slot * STAGE_BYTES;
    uint4 wv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
        if (active && jj < BPS) wv[jj] = *reinterpret_cast<const uint4 *>(base + woff[jj]);
    const int b0 = sub * BPS;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < m) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                dst[t][jj] = MAGIC_I;
                if (active && jj < BPS) {
                    const int xb = t * NB + b0 + ((jj + rot) & (BPS - 1));
                    dst[t][jj] = block_dot_i(wv[jj], xlo[xb], xhi[xb], xcb[xb]);
                }
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    ++it;
    return true;
}

// In-order F32 fold of one stage into acc: lane 0 of the quad folds its
// sub-chunk's blocks, hands the running sum to lane 1, and so on.  dx points
// at the scales of the stage's first block (token 0).
template <int MT>
__device__ __forceinline__ void stage_fold(const float *dx, int NB, int BPS, int nsub, int m, int q,
                                           int lane, const int (&src)[MT][8], float (&acc)[MT])
{
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < m) {
            float c = acc[t];
#pragma unroll
            for (int l = 0; l < 4; ++l) {
                if (l > 0) c = __shfl_sync(FULL, c, (lane & ~3) | (l - 1));
                if (q == l && l < nsub) {
                    // q == l is a compile-time constant here, so is the rotation
                    const float *dt = dx + t * NB + l * BPS;
                    if (BPS == 8) {
                        const float4 d0 = *reinterpret_cast<const float4 *>(dt);
                        const float4 d1 = *reinterpret_cast<const float4 *>(dt + 4);
                        const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                        for (int b = 0; b < 8; ++b)
                            c = __fmaf_rn(dd[b], __int_as_float(src[t][(b - 2 * l) & 7]) - MAGIC_F, c);
                    } else {
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            c = __fmaf_rn(dt[b], __int_as_float(src[t][(b - 2 * l) & 3]) - MAGIC_F, c);
                    }
                }
            }
            acc[t] = __shfl_sync(FULL, c, (lane & ~3) | 3);
        }
    }
}

// Largest of 4, 2, 1 dividing n.
__device__ __forceinline__ int nsub_for(int n) { return (n % 4 == 0) ? 4 : (n % 2 == 0) ? 2 : 1; }

// MT: bound on the tokens of any tile in this launch (1, 2 or 4; <= GEMV_MT).
template <int MT>
__global__ void __launch_bounds__(EXPERT_THREADS, 1)
k_experts(const __grid_constant__ ExpertMaps maps, const ExpertArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *ring = smem;
    const int NBmax = (a.H > a.F ? a.H : a.F) / 32;
    uint4 *xlo = reinterpret_cast<uint4 *>(ring + NSTAGE * STAGE_BYTES);
    uint4 *xhi = xlo + GEMV_MT * NBmax;
    int *xcb = reinterpret_cast<int *>(xhi + GEMV_MT * NBmax);
    float *xd = reinterpret_cast<float *>(xcb + GEMV_MT * NBmax);
    float *red = xd + GEMV_MT * NBmax;
    ExpertSmem &S = *reinterpret_cast<ExpertSmem *>(red + GEMV_MT * 64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, F = a.F, KC = a.KC;
    const int G = F / 32, CH = H / 64;
    const int n_tiles = *a.n_tiles;
    // sub-chunks per stage and stages per unit, for gate/up (K = H) and down (K = F)
    const int nsub_gu = nsub_for((H / 2) / KC), nsub_dn = nsub_for((F / 2) / KC);
    const int nst_gu = (H / 2) / (KC * nsub_gu), nst_dn = (F / 2) / (KC * nsub_dn);
    // static schedule: this block's share of the gate/up units, then of the down units
    const long NG = (long)n_tiles * G, NW = a.gate_up_only ? 0 : (long)n_tiles * CH;
    const long g0 = NG * blockIdx.x / gridDim.x, g1 = NG * (blockIdx.x + 1) / gridDim.x;
    const long w0 = NW * blockIdx.x / gridDim.x, w1 = NW * (blockIdx.x + 1) / gridDim.x;
    const long n_units = (g1 - g0) + (w1 - w0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], CONSUMER_WARPS);
        }
        S.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CONSUMER_WARPS) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            prefetch_tmap(&maps.gu);
            prefetch_tmap(&maps.dn);
            prefetch_tmap(&maps.sgu);
            prefetch_tmap(&maps.sdn);
            const uint64_t pol = policy_evict_first();
            long it = 0;
            for (long i = 0; i < n_units && !S.abort; ++i) {
                const bool gu = i < g1 - g0;
                const long v = gu ? g0 + i : w0 + (i - (g1 - g0));
                const int tile = (int)(gu ? v / G : v / CH);
                const int j = (int)(gu ? v - (long)tile * G : v - (long)tile * CH);
                const int e = __ldg(a.tile_expert + tile);
                const bool shared = (e == a.E);
                const int z = shared ? 0 : e;
                const int nst = gu ? nst_gu : nst_dn, nsub = gu ? nsub_gu : nsub_dn;
                const void *m = gu ? (shared ? (const void *)&maps.sgu : (const void *)&maps.gu)
                                   : (shared ? (const void *)&maps.sdn : (const void *)&maps.dn);
                for (int s = 0; s < nst; ++s, ++it) {
                    const int slot = (int)(it % NSTAGE);
                    const uint32_t round = (uint32_t)(it / NSTAGE);
                    if (round > 0 && !mbar_wait_bounded(&S.empty[slot], (round - 1) & 1)) {
                        set_status(a.status, ST_TIMEOUT);
                        S.abort = 1;
                        break;
                    }
                    unsigned char *dst = ring + slot * STAGE_BYTES;
                    mbar_arrive_expect_tx(&S.full[slot], STAGE_ROWS * KC * nsub);
                    for (int c = 0; c < nsub; ++c) {
                        const int x = (s * nsub + c) * KC;
                        unsigned char *d = dst + c * SUB_BYTES;
                        if (gu) {
                            tma_load_3d(d, m, x, 32 * j, z, &S.full[slot], pol);
                            tma_load_3d(d + 32 * KC, m, x, F + 32 * j, z, &S.full[slot], pol);
                        } else {
                            tma_load_3d(d, m, x, 64 * j, z, &S.full[slot], pol);
                        }
                    }
                }
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int r = 8 * warp + (lane >> 2);     // weight row of the stage owned by this lane's quad
    const int q = lane & 3;                   // sub-chunk owned by this lane
    const int BPS = KC / 16;                  // 32-weight blocks per sub-chunk row (8 or 4)
    const bool swz = (KC == 128);
    // Visiting order rotated by 2q blocks keeps the four lanes of a quad on
    // distinct shared-memory banks: slot jj of this lane holds block (jj + rot).
    const int rot = (2 * q) & (BPS - 1);
    int woff[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
        const int blk = (jj + rot) & (BPS - 1);
        woff[jj] = q * SUB_BYTES + r * KC + 16 * (swz ? (blk ^ (r & 7)) : blk);
    }

    long it = 0;
    int staged_tile = -1;
    bool staged_gu = false;
    bool aborted = false;
    for (long i = 0; i < n_units && !aborted; ++i) {
        const bool gu = i < g1 - g0;
        const long v = gu ? g0 + i : w0 + (i - (g1 - g0));
        const int tile = (int)(gu ? v / G : v / CH);
        const int j = (int)(gu ? v - (long)tile * G : v - (long)tile * CH);
        const int e = __ldg(a.tile_expert + tile);
        const int pos0 = __ldg(a.tile_pos0 + tile);
        const int m = __ldg(a.tile_m + tile);
        const int nst = gu ? nst_gu : nst_dn, nsub = gu ? nsub_gu : nsub_dn;
        const int NB = gu ? H / 32 : F / 32;
        const float *ers = (e == a.E) ? a.shared_rs : a.expert_rs + (size_t)e * (2 * F + H);
        const bool active = q < nsub;

        if (tile != staged_tile || gu != staged_gu) {
            // activations of the tile: x codes for gate/up, h codes for down
            if (threadIdx.x == 0) {
                if (!gu) {
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire_gpu(&a.g_done[tile]) < G) {
                        if (globaltimer() - t0 > WAIT_NS) {
                            set_status(a.status, ST_TIMEOUT);
                            break;
                        }
                        nanosleep_ns(32);
                    }
                }
                for (int t = 0; t < MT; ++t)
                    S.tok[t] = (t < m) ? (gu ? __ldg(a.pos_token + pos0 + t) : pos0 + t) : 0;
            }
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (gu)
                stage_acts(a.qx, a.dx, H, m, S.tok, a.n_tok, xlo, xhi, xcb, xd, a.status);
            else
                stage_acts(a.qh, a.dh, F, m, S.tok, a.P + a.n_tok, xlo, xhi, xcb, xd, a.status);
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            staged_tile = tile;
            staged_gu = gu;
        }

        // Software pipeline over the unit's stages: the integer block dots of
        // stage s+1 are issued next to the in-order F32 fold of stage s, and a
        // ring slot is released as soon as its integer dots are done.
        float acc[MT];
        int Ic[MT][8];   // stage being folded: biased block dots (MAGIC_I + I)
        int In[MT][8];   // next stage
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.0f;

        // ping-pong between the two buffers, two stages per iteration
#define COLI_DOTS(s_, dst_)                                                                     \
    stage_dots<MT>(S.full, S.empty, ring, it, woff, xlo, xhi, xcb, (s_) * nsub + q, BPS, rot, NB, \
                   m, active, lane, dst_)
#define COLI_FOLD(s_, src_) \
    stage_fold<MT>(xd + (s_) * nsub * BPS, NB, BPS, nsub, m, q, lane, src_, acc)
        if (!COLI_DOTS(0, Ic)) { aborted = true; break; }
        for (int s = 0; s < nst; s += 2) {
            if (s + 1 < nst && !COLI_DOTS(s + 1, In)) { aborted = true; break; }
            COLI_FOLD(s, Ic);
            if (s + 1 >= nst) break;
            if (s + 2 < nst && !COLI_DOTS(s + 2, Ic)) { aborted = true; break; }
            COLI_FOLD(s + 1, In);
        }
#undef COLI_DOTS
#undef COLI_FOLD
        if (aborted) break;

        // ---- unit epilogue ----
        if (gu) {
            if (q == 0)
                for (int t = 0; t < m; ++t) red[t * 64 + r] = acc[t];
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (warp < m) {
                const int t = warp, ii = 32 * j + lane, pos = pos0 + t;
                const float gg = __fmul_rn(ers[ii], red[t * 64 + lane]);
                const float uu = __fmul_rn(ers[F + ii], red[t * 64 + 32 + lane]);
                const float h = __fmul_rn(__fmul_rn(gg, own_sigmoid(gg)), uu);
                float dq;
                const int qv = q8_0_lane(h, &dq);
                a.qh[(size_t)pos * F + ii] = (int8_t)qv;
                if (lane == 0) a.dh[(size_t)pos * G + j] = dq;
                if (a.h_dbg) a.h_dbg[(size_t)pos * F + ii] = h;
            }
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (threadIdx.x == 0) red_release_gpu(&a.g_done[tile], 1);
        } else {
            const int row = 64 * j + r;
            if (q == 0)
                for (int t = 0; t < m; ++t)
                    a.y[(size_t)(pos0 + t) * H + row] = __fmul_rn(ers[2 * F + row], acc[t]);
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (threadIdx.x == 0) red_release_gpu(&a.w_done[j], 1);
        }
    }

    if (aborted) {
        set_status(a.status, ST_TIMEOUT);
        S.abort = 1;
        // wait (bounded) for copies still in flight into this block's ring
        // before the block exits
        if (threadIdx.x == 0)
            for (int i = 0; i < NSTAGE; ++i, ++it)
                (void)mbar_wait_bounded(&S.full[(int)(it % NSTAGE)], (uint32_t)(it / NSTAGE) & 1);
        return;
    }

    // ---- combine: this block owns the chunks whose last-tile down unit it ran ----
    if (!a.gate_up_only && n_tiles > 0) {
        const long last0 = (long)(n_tiles - 1) * CH;
        const long c0 = (w0 > last0 ? w0 : last0) - last0;
        const long c1 = (w1 > last0 ? w1 : last0) - last0;
        const int T = a.n_tok, k = a.k, P = a.P;
        for (long c = c0; c < c1; ++c) {
            if (threadIdx.x == 0) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_gpu(&a.w_done[c]) < n_tiles) {
                    if (globaltimer() - t0 > WAIT_NS) {
                        set_status(a.status, ST_TIMEOUT);
                        break;
                    }
                    nanosleep_ns(32);
                }
            }
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            for (int ii = threadIdx.x; ii < T * 64; ii += CONSUMERS) {
                const int t = ii >> 6, col = 64 * (int)c + (ii & 63);
                float o = __ldcg(a.y + (size_t)(P + t) * H + col);
                for (int rr = 0; rr < k; ++rr) {
                    const int pos = __ldcg(a.inv + (size_t)t * k + rr);
                    if (pos < 0 || pos >= P) continue;
                    o = __fmaf_rn(__ldcg(a.wts + (size_t)t * k + rr), __ldcg(a.y + (size_t)pos * H + col), o);
                }
                a.out[(size_t)t * H + col] = o;
            }
        }
    }
}

template <int MT>
static int launch_experts_mt(const ExpertMaps &maps, const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    static size_t configured = 0;
    const size_t smem = experts_smem_bytes(a.H, a.F);
    if (smem != configured) {
        if (cudaFuncSetAttribute(k_experts<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return -1;
        configured = smem;
    }
    k_experts<MT><<<num_sms, EXPERT_THREADS, smem, st>>>(maps, a);
    count_launch();
    return 0;
}

int launch_experts(const ExpertMaps &maps, const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    // tiles hold at most min(T, GEMV_MT) tokens
    const int mt = a.n_tok < GEMV_MT ? a.n_tok : GEMV_MT;
    if (mt <= 1) return launch_experts_mt<1>(maps, a, num_sms, st);
    if (mt <= 2) return launch_experts_mt<2>(maps, a, num_sms, st);
    return launch_experts_mt<4>(maps, a, num_sms, st);
}

}  // namespace coli
