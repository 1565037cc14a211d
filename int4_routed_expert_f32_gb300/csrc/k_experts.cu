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
// Structure: several small blocks per SM, each 2 consumer warps + 1 producer
// warp, all blocks resident (the grid is sized by the occupancy calculator).
//   * Work units, claimed in increasing order (block b starts with unit b,
//     then takes the next one from a global counter with the current unit's
//     last copy): first
//     every gate/up unit (a tile of <= GEMV_MT tokens of one expert x 32
//     hidden units = 32 gate rows + 32 up rows), then every down unit (a tile x
//     64 output rows).
//   * The producer streams a unit's 64 weight rows through a ring of stages
//     with 3-D TMA tile loads: a stage is 64 rows x 256 bytes (512 weights of
//     each row) as two swizzled boxes of 64 rows x 128 bytes (128-byte
//     swizzle), L2 evict-first.  Each stage completes on its mbarrier; the
//     consumers release it through a second one.
//   * Consumer lane r owns weight row r: per stage it reads its row's 16
//     blocks of 32 weights (the swizzle keeps the 32 lanes on distinct banks),
//     does the dp4a block dots and folds them into its F32 accumulator in
//     block order, acc = fma(d_b, I_b, acc): the row's whole dot product lives
//     in one lane, so the order is the fixed ascending one without any
//     exchange.  Sixteen independent block dots per stage give each warp
//     enough instruction-level parallelism; a few blocks per SM hide the rest.
//   * A down unit needs the h codes of its whole tile: it waits (bounded) on
//     the tile's gate/up completion counter.  The block that finishes the last
//     down unit of a 64-row output chunk (over all tiles) combines the chunk.
//   * Launched as a programmatic dependent of the routing kernel: set-up
//     overlaps routing, and every thread waits for the routing grid
//     (griddepcontrol.wait) before reading its results.  The counters start at
//     zero (configure) and the last block to exit zeroes them for the next
//     launch.
#include <cstdlib>

#include <cuda.h>

#include "coli_common.cuh"
#include "coli_internal.h"
#include "tma.cuh"

namespace coli {

constexpr int NSTAGE_MAX = 6;
constexpr int STAGE_ROWS = 64;
constexpr int KC_MAX = 128;
constexpr int NSUB_MAX = 2;                        // TMA boxes along K per stage
constexpr int SUB_BYTES = STAGE_ROWS * KC_MAX;     // 8 KB: one box of 64 rows x 128 B
constexpr int STAGE_BYTES = NSUB_MAX * SUB_BYTES;  // 16 KB
constexpr int BAR_CONSUMERS = 1;                   // named barrier id (0 = __syncthreads)

// Consumer warps of a block: two (lane r of warp w owns weight row 32w + r of
// each stage) for one-token tiles; four for multi-token tiles, where each pair
// of warps takes half of the tile's tokens over the same 64 rows.  Multi-token
// tiles are bound by the block dots' issue rate (each weight feeds a dp4a
// chain per token), so twice the warps issue them, with no exchange between
// the pairs: every (row, token) fold stays in one lane.
template <int MT> struct Cons {
    static constexpr int WARPS = MT >= 2 ? 4 : 2;
    static constexpr int N = WARPS * 32;            // consumer threads
    static constexpr int THREADS = N + 32;          // and the producer warp
    static constexpr int PAIRS = WARPS / 2;
    static constexpr int TP = MT / PAIRS;           // tokens per pair
    // three blocks per SM (as shared memory allows): for the 160-thread blocks
    // this bounds the registers to 136
    static constexpr int MIN_BLOCKS = 3;
};
constexpr uint64_t WAIT_NS = 2000000000ull;        // 2 s bound on every ring wait

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


// Optional event log: per block, trace_cap slots of (globaltimer << 8 | code)
// followed by the unit; slot 0 counts the events.  Codes: 1 kernel start,
// 2 unit start (first stage arrived), 3 activations staged, 4 unit done,
// 5 combine done, 6 consumer exit, 7 consumer time waiting for data (the
// unit field holds nanoseconds); the producer's waiting time for free ring
// slots is code 8 in the block's last slot.
__device__ __forceinline__ void trace_event(const ExpertArgs &a, int code, long unit)
{
    if (!a.trace || threadIdx.x != 0) return;
    unsigned long long *blk = a.trace + (size_t)blockIdx.x * a.trace_cap * 2;
    const unsigned long long n = blk[0];
    if ((long)n + 1 >= a.trace_cap) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    blk[2 * (n + 1)] = (t << 8) | (unsigned)code;
    blk[2 * (n + 1) + 1] = (unsigned long long)unit;
    blk[0] = n + 1;
}

// Bounded spin until *p >= target; false if it gave up after bound_ns.
__device__ __forceinline__ bool wait_counter(const int *p, int target, uint64_t bound_ns)
{
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(p) < target) {
        if (globaltimer() - t0 > bound_ns) return false;
        nanosleep_ns(64);
    }
    return true;
}

struct ExpertSmem {
    int stage_unit[NSTAGE_MAX];     // unit of each ring slot (-1: no more work)
    int stage_k[NSTAGE_MAX];        // stage index inside the unit
    int abort;
    int combine;
    int tok[GEMV_MT];               // rows of the activations being staged
    alignas(8) uint64_t full[NSTAGE_MAX];
    alignas(8) uint64_t empty[NSTAGE_MAX];
};

static size_t act_bytes(int H, int F, int mt)
{
    const int NB = (H > F ? H : F) / 32;
    return (size_t)mt * NB * (16 + 16 + 4 + 4);
}

size_t experts_smem_bytes_mt(int H, int F, int mt, int nstage)
{
    // no alignment slack: the kernel takes its dynamic shared memory at a
    // 1024-byte boundary (checked at its start), which lets four one-token
    // blocks of the decode layer share an SM
    return (size_t)nstage * STAGE_BYTES + act_bytes(H, F, mt) +
           (size_t)mt * 32 * 4 + sizeof(ExpertSmem);
}

// Ring depth.  More blocks per SM help more than deeper rings.  Three stages,
// unless three blocks of that size do not fit in one SM's shared memory
// (several tokens' activations make the block larger); then two, which keeps
// three blocks per SM (a 4-token forward ran 26% faster that way).  The
// one-token decode layer's 3-stage blocks fit four per SM, which runs every
// gate/up unit of a forward in the first wave.  COLI_MOE_RING_STAGES (2..6)
// overrides the choice for tuning.
static int ring_stages(int H, int F, int mt)
{
    static int env_n = -1;
    if (env_n < 0) {
        const char *env = getenv("COLI_MOE_RING_STAGES");
        const int v = env ? atoi(env) : 0;
        env_n = (v >= 2 && v <= NSTAGE_MAX) ? v : 0;
    }
    if (env_n > 0) return env_n;
    static int smem_per_sm = 0;
    if (smem_per_sm == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess && v > 0)
            smem_per_sm = v;
        else
            smem_per_sm = 228 * 1024;
    }
    // 1 KB of each block's shared memory is reserved by the system
    return 3 * (experts_smem_bytes_mt(H, F, mt, 3) + 1024) <= (size_t)smem_per_sm ? 3 : 2;
}

size_t experts_smem_bytes(int H, int F) { return experts_smem_bytes_mt(H, F, GEMV_MT, ring_stages(H, F, GEMV_MT)); }

// Activations of one tile into shared memory, xlo/xhi/xcd [MT][NB].  For
// int4 weights (WB = 4) the codes are held in split form (see block_dot) and
// xcd holds (MAGIC_I - 8 * sum of the codes, the block's F32 scale bits), the
// nibble offset folded in; for int8 weights (WB = 8) xlo/xhi hold the block's
// codes 0..15 and 16..31 as they are and xcd (MAGIC_I, scale bits).  One
// 8-byte load serves both halves of xcd.  Loads are issued SU at a time per
// thread so that a tile's staging costs about one L2 round trip.
template <int MT, int WB>
__device__ __forceinline__ void stage_acts(const int8_t *__restrict__ q, const float *__restrict__ d,
                                           int K, int m, const int *rows, int row_limit,
                                           uint4 *xlo, uint4 *xhi, int2 *xcd, int *status)
{
    constexpr int SU = 4;
    constexpr int CONSUMERS = Cons<MT>::N;
    const int NB = K / 32;
    for (int i0 = threadIdx.x; i0 < MT * NB; i0 += CONSUMERS * SU) {
        uint4 va[SU], vb[SU];
        float vd[SU];
#pragma unroll
        for (int uu = 0; uu < SU; ++uu) {
            const int i = i0 + uu * CONSUMERS;
            va[uu] = vb[uu] = make_uint4(0, 0, 0, 0);
            vd[uu] = 0.0f;
            if (i < MT * NB) {
                const int t = i / NB, b = i - t * NB;
                if (t < m) {
                    const int row = rows[t];
                    if (row >= 0 && row < row_limit) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(q + (size_t)row * K + (size_t)b * 32);
                        va[uu] = __ldcg(src);
                        vb[uu] = __ldcg(src + 1);
                        vd[uu] = __ldcg(d + (size_t)row * NB + b);
                    } else {
                        set_status(status, ST_BAD_INDEX);
                    }
                }
            }
        }
#pragma unroll
        for (int uu = 0; uu < SU; ++uu) {
            const int i = i0 + uu * CONSUMERS;
            if (i < MT * NB) {
                if (WB == 4) {
                    uint4 lo, hi;
                    int sum;
                    split_block(va[uu], vb[uu], &lo, &hi, &sum);
                    xlo[i] = lo;
                    xhi[i] = hi;
                    xcd[i] = make_int2(MAGIC_I - 8 * sum, __float_as_int(vd[uu]));
                } else {
                    xlo[i] = va[uu];
                    xhi[i] = vb[uu];
                    xcd[i] = make_int2(MAGIC_I, __float_as_int(vd[uu]));
                }
            }
        }
    }
}

// Integer dot of a block with the low and high nibbles accumulated apart:
// the high nibbles are used in place (16 x nibble), so no shifts are needed.
// Returns MAGIC_I + I when cb = MAGIC_I - 8 * sum(x).
__device__ __forceinline__ int block_dot_i(uint4 w, uint4 lo, uint4 hi, int cb)
{
    // four short chains instead of two long ones
    int a0 = dp4a_us(w.x & 0x0F0F0F0Fu, (int)lo.x, cb);
    int a1 = dp4a_us(w.y & 0x0F0F0F0Fu, (int)lo.y, 0);
    int h0 = dp4a_us(w.x & 0xF0F0F0F0u, (int)hi.x, 0);
    int h1 = dp4a_us(w.y & 0xF0F0F0F0u, (int)hi.y, 0);
    a0 = dp4a_us(w.z & 0x0F0F0F0Fu, (int)lo.z, a0);
    a1 = dp4a_us(w.w & 0x0F0F0F0Fu, (int)lo.w, a1);
    h0 = dp4a_us(w.z & 0xF0F0F0F0u, (int)hi.z, h0);
    h1 = dp4a_us(w.w & 0xF0F0F0F0u, (int)hi.w, h1);
    return (a0 + a1) + ((h0 + h1) >> 4);
}

// Integer dot of a block of 32 int8 weights (two 16-byte chunks) with the
// block's 32 int8 codes (xlo: codes 0..15, xhi: 16..31).  Returns MAGIC_I + I
// when cb = MAGIC_I (|I| <= 32 * 127 * 127 < 2^22).
__device__ __forceinline__ int block_dot_i8(uint4 w0, uint4 w1, uint4 lo, uint4 hi, int cb)
{
    int a0 = __dp4a((int)w0.x, (int)lo.x, cb);
    int a1 = __dp4a((int)w0.y, (int)lo.y, 0);
    int a2 = __dp4a((int)w0.z, (int)lo.z, 0);
    int a3 = __dp4a((int)w0.w, (int)lo.w, 0);
    a0 = __dp4a((int)w1.x, (int)hi.x, a0);
    a1 = __dp4a((int)w1.y, (int)hi.y, a1);
    a2 = __dp4a((int)w1.z, (int)hi.z, a2);
    a3 = __dp4a((int)w1.w, (int)hi.w, a3);
    return (a0 + a1) + (a2 + a3);
}

// One stage for this lane's row: the NSUB x BPS block dots of every token,
// then their in-order fold into acc.  A block is one 16-byte chunk of the
// row for int4 weights, two for int8 (CPB chunks per block; woff holds the
// row's eight chunk offsets in the box).  All trip counts are compile-time
// constants, so the block dots form one straight-line region the scheduler
// can interleave.
template <int TP, int NSUB, int BPS, int WB>
__device__ __forceinline__ void stage_rows(const unsigned char *base, const int (&woff)[8], const uint4 *xlo,
                                           const uint4 *xhi, const int2 *xcd, int NB, int b0, int t0, int m,
                                           float (&acc)[TP])
{
    constexpr int CPB = WB == 4 ? 1 : 2;
    // One token: the whole stage's bytes in registers, then its block dots
    // and fold.  Several tokens: one box (half a stage) at a time, every
    // token's dots and fold for it, then the next box -- each token still
    // folds its blocks in ascending order, and the row's bytes are loaded
    // once for all tokens without holding the whole stage in registers.
    constexpr int NCH = TP == 1 ? NSUB : 1;      // boxes whose bytes are held at once
#pragma unroll
    for (int c0 = 0; c0 < NSUB; c0 += NCH) {
        uint4 wv[NCH][BPS][CPB];
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int jj = 0; jj < BPS; ++jj)
#pragma unroll
                for (int p = 0; p < CPB; ++p)
                    wv[c][jj][p] =
                        *reinterpret_cast<const uint4 *>(base + (c0 + c) * SUB_BYTES + woff[jj * CPB + p]);
#pragma unroll
        for (int tt = 0; tt < TP; ++tt) {
            const int t = t0 + tt;
            if (t < m) {
                const int xb0 = t * NB + b0 + c0 * BPS;
                int I[NCH][BPS];
                float dd[NCH][BPS];
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int jj = 0; jj < BPS; ++jj) {
                        const int xb = xb0 + c * BPS + jj;
                        const int2 cd = xcd[xb];
                        if (WB == 4)
                            I[c][jj] = block_dot_i(wv[c][jj][0], xlo[xb], xhi[xb], cd.x);
                        else
                            I[c][jj] = block_dot_i8(wv[c][jj][0], wv[c][jj][CPB - 1], xlo[xb], xhi[xb], cd.x);
                        dd[c][jj] = __int_as_float(cd.y);
                    }
                float cacc = acc[tt];
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int jj = 0; jj < BPS; ++jj)
                        cacc = __fmaf_rn(dd[c][jj], __int_as_float(I[c][jj]) - MAGIC_F, cacc);
                acc[tt] = cacc;
            }
        }
    }
}

// L2 prefetch of [lo, hi) clipped to a region of `bytes` bytes (offsets and
// sizes multiples of 16, the base 16-byte aligned).
__device__ __forceinline__ void prefetch_part(const unsigned char *base, size_t bytes, size_t lo, size_t hi)
{
    if (!base || lo >= bytes) return;
    if (hi > bytes) hi = bytes;
    for (size_t o = lo; o < hi; o += 16384) {
        const size_t n = hi - o < 16384 ? hi - o : 16384;
        prefetch_l2_bulk(base + o, (uint32_t)n);
    }
}

// Decode unit u: gate/up units first (tile-major), then down units.
__device__ __forceinline__ void decode_unit(long u, long n_gu, int G, int CH, bool *gu, int *tile, int *j)
{
    *gu = u < n_gu;
    const long v = *gu ? u : u - n_gu;
    const int per = *gu ? G : CH;
    *tile = (int)(v / per);
    *j = (int)(v - (long)*tile * per);
}

// MT: bound on the tokens of any tile in this launch (1, 2 or 4; <= GEMV_MT).
// BPS: 32-weight blocks per box row of KC bytes (int4: 8, 4 or 1 for KC =
// 128, 64 or 16; int8: 4, 2 or 1 for KC = 128, 64 or 32).
// WB: weight container, 4 (packed nibbles) or 8 (one int8 code per byte).
template <int MT, int BPS, int WB>
__global__ void __launch_bounds__(Cons<MT>::THREADS, Cons<MT>::MIN_BLOCKS)
k_experts(const __grid_constant__ ExpertMaps maps, const ExpertArgs a)
{
    constexpr int CONSUMER_WARPS = Cons<MT>::WARPS;
    constexpr int CONSUMERS = Cons<MT>::N;
    constexpr int TP = Cons<MT>::TP;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // The swizzled TMA boxes need 1024-byte alignment, and the size computed
    // on the host has no slack for realigning: a block whose dynamic shared
    // memory starts elsewhere reports ST_BAD_SHAPE and does nothing (every
    // block of a launch sees the same offset).
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(a.status, ST_BAD_SHAPE);
        return;
    }
    unsigned char *smem = smem_raw;
    unsigned char *ring = smem;
    const int NBmax = (a.H > a.F ? a.H : a.F) / 32;
    const int nstage = a.nstage;
    uint4 *xlo = reinterpret_cast<uint4 *>(ring + nstage * STAGE_BYTES);
    uint4 *xhi = xlo + MT * NBmax;
    int2 *xcd = reinterpret_cast<int2 *>(xhi + MT * NBmax);
    float *red = reinterpret_cast<float *>(xcd + MT * NBmax);     // [MT][32] up-row sums
    ExpertSmem &S = *reinterpret_cast<ExpertSmem *>(red + MT * 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, F = a.F, KC = a.KC;
    const int G = F / 32, CH = H / 64;
    // bytes of a gate/up and of a down row; boxes along K per stage (2 when
    // the row's box count is even)
    const int rb_gu = H * WB / 8, rb_dn = F * WB / 8;
    const int nsub_gu = ((rb_gu / KC) % 2 == 0) ? 2 : 1, nsub_dn = ((rb_dn / KC) % 2 == 0) ? 2 : 1;
    const int nst_gu = rb_gu / (KC * nsub_gu), nst_dn = rb_dn / (KC * nsub_dn);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstage; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], CONSUMER_WARPS);
        }
        S.abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * CONSUMER_WARPS) {
        prefetch_tmap(&maps.gu);
        prefetch_tmap(&maps.dn);
        prefetch_tmap(&maps.sgu);
        prefetch_tmap(&maps.sdn);
    }
    // The shared expert runs on every token whatever the routing: while the
    // routing grid is still running, the blocks spread an L2 prefetch of its
    // packed weights over themselves, so that its units read from L2 and HBM
    // does not sit idle during routing.
    if (a.shared_w4 && threadIdx.x == 32 * CONSUMER_WARPS) {
        const size_t total_b = (size_t)3 * F * H * WB / 8;      // multiple of 16 (H % 128, F % 32 == 0)
        const size_t per = ((total_b / gridDim.x) + 4095) & ~(size_t)4095;
        const size_t b0 = (size_t)blockIdx.x * per;
        const size_t b1 = b0 + per < total_b ? b0 + per : total_b;
        for (size_t o = b0; o < b1; o += 16384) {
            const size_t n = b1 - o < 16384 ? b1 - o : 16384;
            prefetch_l2_bulk(a.shared_w4 + o, (uint32_t)n);
        }
    }
    __syncthreads();
    // routing results (tile list, activations) are complete past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_tiles = *a.n_tiles;
    const long n_gu = (long)n_tiles * G;
    const long total = a.gate_up_only ? n_gu : n_gu + (long)n_tiles * CH;

    if (warp == CONSUMER_WARPS) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            unsigned long long waited = 0;      // traced: time spent waiting for free slots
            int slot = 0;
            uint32_t phase = 0;       // parity of the ring's current round
            bool first_round = true;
            // every block is resident: the first unit of block b is unit b
            // (no atomic round trip at the start), later claims come from
            // the counter, offset by the grid
            long u = blockIdx.x;
            for (;;) {
                const bool done = u >= total || S.abort;
                bool gu = false;
                int tile = 0, j = 0, e = 0;
                if (!done) {
                    decode_unit(u, n_gu, G, CH, &gu, &tile, &j);
                    e = __ldg(a.tile_expert + tile);
                }
                long u_next = total;
                const int nst = done ? 1 : (gu ? nst_gu : nst_dn);
                const int nsub = gu ? nsub_gu : nsub_dn;
                const bool shared = (e == a.E);
                const void *m = gu ? (shared ? (const void *)&maps.sgu : (const void *)&maps.gu)
                                   : (shared ? (const void *)&maps.sdn : (const void *)&maps.dn);
                const int z = shared ? 0 : (a.slot_of ? __ldg(a.slot_of + e) : e);
                bool stop = false;
                for (int s = 0; s < nst; ++s) {
                    const unsigned long long w0 = a.trace ? globaltimer() : 0;
                    const bool got = first_round || mbar_wait_bounded(&S.empty[slot], phase ^ 1);
                    if (a.trace) waited += globaltimer() - w0;
                    if (!got) {
                        set_status(a.status, ST_TIMEOUT);
                        S.abort = 1;
                        stop = true;
                    }
                    if (done || stop) {
                        S.stage_unit[slot] = -1;
                        mbar_arrive(&S.full[slot]);
                        stop = true;
                        break;
                    }
                    S.stage_unit[slot] = (int)u;
                    S.stage_k[slot] = s;
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
                    if (++slot == nstage) {
                        slot = 0;
                        phase ^= 1;
                        first_round = false;
                    }
                    // claim the next unit with this unit's last copy: the
                    // atomic's round trip overlaps the stages still in the
                    // ring, and units are handed out in the order in which
                    // blocks run out of work (claimed at the start of a unit,
                    // a block's second unit was fixed before its first ran)
                    if (s == nst - 1) u_next = (long)gridDim.x + atomicAdd(a.work_counter, 1);
                }
                if (stop) break;
                u = u_next;
            }
            // Layer-ahead prefetch (stacked decode): a block with no unit
            // left pulls its share of the next layer's router weights and
            // shared expert into L2.  Neither depends on the next layer's
            // routing, and HBM is partly idle while the rest of the grid
            // finishes this layer's last down units.
            if ((a.next_rw || a.next_sw) && !S.abort) {
                const size_t total_b = a.next_rw_bytes + a.next_sw_bytes;
                const size_t per = ((total_b / gridDim.x) + 4095) & ~(size_t)4095;
                const size_t lo = (size_t)blockIdx.x * per, hi = lo + per;
                prefetch_part(a.next_rw, a.next_rw_bytes, lo, hi);
                if (hi > a.next_rw_bytes)
                    prefetch_part(a.next_sw, a.next_sw_bytes, lo > a.next_rw_bytes ? lo - a.next_rw_bytes : 0,
                                  hi - a.next_rw_bytes);
            }
            if (a.trace) {
                // the producer's lane logs its waiting time in the block's last slot
                unsigned long long *blk = a.trace + (size_t)blockIdx.x * a.trace_cap * 2;
                blk[2 * (a.trace_cap - 1)] = (waited << 8) | 8u;
                blk[2 * (a.trace_cap - 1) + 1] = 0;
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int r = threadIdx.x & 63;           // this lane's weight row in the stage (0..63)
    const int t0 = (threadIdx.x >> 6) * TP;   // this pair's first token of a tile
    const int half = warp & 1;                // rows 0..31 (gate rows of a gate/up unit) or 32..63
    const bool swz = (KC == 128);
    int woff[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) woff[jj] = r * KC + 16 * (swz ? (jj ^ (r & 7)) : jj);

    int slot = 0;
    uint32_t phase = 0;
    int staged_tile = -1;            // tile whose h codes are staged (down units)
    int staged_tok[GEMV_MT];         // tokens whose x codes are staged (gate/up units)
    int staged_m = -1;
#pragma unroll
    for (int t = 0; t < GEMV_MT; ++t) staged_tok[t] = -1;
    trace_event(a, 1, -1);
    float acc[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) acc[t] = 0.0f;
    bool gu = true;
    int tile = 0, j = 0, e = 0, pos0 = 0, m = 0, nst = 0, NB = 0, nsub = 1;
    const float *ers = nullptr;

    unsigned long long full_wait = 0;    // traced: time spent waiting for filled slots
    for (;;) {
        const unsigned long long fw0 = a.trace ? globaltimer() : 0;
        const bool got = mbar_wait_bounded(&S.full[slot], phase);
        if (a.trace) full_wait += globaltimer() - fw0;
        if (!got) {
            set_status(a.status, ST_TIMEOUT);
            S.abort = 1;
            break;
        }
        const int u = S.stage_unit[slot];
        const int s = S.stage_k[slot];
        if (u < 0) break;
        if (s == 0) {
            // new unit
            trace_event(a, 2, u);
            decode_unit(u, n_gu, G, CH, &gu, &tile, &j);
            e = __ldg(a.tile_expert + tile);
            pos0 = __ldg(a.tile_pos0 + tile);
            m = __ldg(a.tile_m + tile);
            nst = gu ? nst_gu : nst_dn;
            nsub = gu ? nsub_gu : nsub_dn;
            NB = gu ? H / 32 : F / 32;
            ers = (e == a.E) ? a.shared_rs
                             : a.expert_rs + (size_t)(a.slot_of ? __ldg(a.slot_of + e) : e) * (2 * F + H);
            // activations: x codes of the tile's tokens for gate/up (kept while
            // the token set is unchanged), h codes of the tile for down
            bool restage;
            if (gu) {
                restage = (m != staged_m) || staged_tile >= 0;
#pragma unroll
                for (int t = 0; t < GEMV_MT; ++t)
                    if (t < m && __ldg(a.pos_token + pos0 + t) != staged_tok[t]) restage = true;
            } else {
                restage = (tile != staged_tile);
            }
            if (restage) {
                if (threadIdx.x == 0) {
                    if (!gu && !wait_counter(&a.g_done[tile], G + a.gdone_extra, a.wait_ns))
                        set_status(a.status, ST_TIMEOUT);
                    for (int t = 0; t < GEMV_MT; ++t)
                        S.tok[t] = (t < m) ? (gu ? __ldg(a.pos_token + pos0 + t) : pos0 + t) : 0;
                }
                named_barrier(BAR_CONSUMERS, CONSUMERS);
                if (gu)
                    stage_acts<MT, WB>(a.qx, a.dx, H, m, S.tok, a.n_tok, xlo, xhi, xcd, a.status);
                else
                    stage_acts<MT, WB>(a.qh, a.dh, F, m, S.tok, a.P + a.n_tok, xlo, xhi, xcd, a.status);
#pragma unroll
                for (int t = 0; t < GEMV_MT; ++t) staged_tok[t] = gu ? S.tok[t] : -1;
                staged_m = gu ? m : -1;
                staged_tile = gu ? -1 : tile;
                named_barrier(BAR_CONSUMERS, CONSUMERS);
                trace_event(a, 3, u);
            }
#pragma unroll
            for (int t = 0; t < TP; ++t) acc[t] = 0.0f;
        }

        // ---- one stage: this lane's row, blocks b0 .. b0 + nsub * BPS - 1, in order ----
        {
            const unsigned char *base = ring + slot * STAGE_BYTES;
            const int b0 = s * nsub * BPS;
            if (nsub == 2)
                stage_rows<TP, 2, BPS, WB>(base, woff, xlo, xhi, xcd, NB, b0, t0, m, acc);
            else
                stage_rows<TP, 1, BPS, WB>(base, woff, xlo, xhi, xcd, NB, b0, t0, m, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        if (++slot == nstage) {
            slot = 0;
            phase ^= 1;
        }
        if (s != nst - 1) continue;

        // ---- unit epilogue ----
        if (gu) {
            // rows 0..31: gate rows 32j.., rows 32..63: the matching up rows;
            // each pair of warps finishes its own tokens
            if (half == 1)
#pragma unroll
                for (int tt = 0; tt < TP; ++tt)
                    if (t0 + tt < m) red[(t0 + tt) * 32 + lane] = acc[tt];
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (half == 0) {
                const int ii = 32 * j + lane;
                const float sg = ers[ii], su = ers[F + ii];
#pragma unroll
                for (int tt = 0; tt < TP; ++tt) {
                    const int t = t0 + tt;
                    if (t < m) {
                        const int pos = pos0 + t;
                        const float gg = __fmul_rn(sg, acc[tt]);
                        const float uu = __fmul_rn(su, red[t * 32 + lane]);
                        const float h = __fmul_rn(__fmul_rn(gg, own_sigmoid(gg)), uu);
                        float dq;
                        const int qv = q8_0_lane(h, &dq);
                        a.qh[(size_t)pos * F + ii] = (int8_t)qv;
                        if (lane == 0) a.dh[(size_t)pos * G + j] = dq;
                        if (a.h_dbg) a.h_dbg[(size_t)pos * F + ii] = h;
                    }
                }
            }
            named_barrier(BAR_CONSUMERS, CONSUMERS);   // h is written; red[] is reused by the next unit
            // every consumer's h stores precede this release (the barrier)
            if (threadIdx.x == 0) red_release_gpu(&a.g_done[tile], 1);
            trace_event(a, 4, u);
        } else {
            const int row = 64 * j + r;
            const float sd = ers[2 * F + row];
#pragma unroll
            for (int tt = 0; tt < TP; ++tt)
                if (t0 + tt < m) a.y[(size_t)(pos0 + t0 + tt) * H + row] = __fmul_rn(sd, acc[tt]);
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (threadIdx.x == 0) {
                __threadfence();
                const int old = atomic_add_acq_rel_gpu(&a.w_done[j], 1);
                S.combine = (old == n_tiles - 1);
            }
            named_barrier(BAR_CONSUMERS, CONSUMERS);
            if (S.combine) {
                // every tile's down rows of this chunk are written: combine them
                __threadfence();
                const int T = a.n_tok, k = a.k, P = a.P;
                for (int ii = threadIdx.x; ii < T * 64; ii += CONSUMERS) {
                    const int t = ii >> 6, col = 64 * j + (ii & 63);
                    float o = __ldcg(a.y + (size_t)(P + t) * H + col);
                    for (int rr = 0; rr < k; ++rr) {
                        const int pos = __ldcg(a.inv + (size_t)t * k + rr);
                        if (pos < 0 || pos >= P) continue;
                        o = __fmaf_rn(__ldcg(a.wts + (size_t)t * k + rr),
                                      __ldcg(a.y + (size_t)pos * H + col), o);
                    }
                    if (a.res) o = __fadd_rn(__ldg(a.res + (size_t)t * H + col), o);
                    a.out[(size_t)t * H + col] = o;
                }
                named_barrier(BAR_CONSUMERS, CONSUMERS);
                trace_event(a, 5, u);
            }
            trace_event(a, 4, u);
        }
    }
    trace_event(a, 6, -1);
    trace_event(a, 7, (long)full_wait);

    if (S.abort && threadIdx.x == 0) {
        // a wait gave up: wait (bounded) for copies still in flight into this
        // block's ring before the block exits
        for (int i = 0; i < nstage; ++i) {
            (void)mbar_wait_bounded(&S.full[slot], phase);
            if (++slot == nstage) {
                slot = 0;
                phase ^= 1;
            }
        }
    }

    // the last block out zeroes the counters for the next launch
    named_barrier(BAR_CONSUMERS, CONSUMERS);
    if (threadIdx.x == 0) {
        __threadfence();
        S.combine = (atomic_add_acq_rel_gpu(a.blocks_done, 1) == (int)gridDim.x - 1);
    }
    named_barrier(BAR_CONSUMERS, CONSUMERS);
    if (S.combine) {
        for (int i = threadIdx.x; i < a.n_sync; i += CONSUMERS)
            if (a.sync_base + i != a.blocks_done) a.sync_base[i] = 0;
        named_barrier(BAR_CONSUMERS, CONSUMERS);
        if (threadIdx.x == 0) {
            __threadfence();
            *a.blocks_done = 0;
        }
    }
}

template <int MT, int BPS, int WB>
static int launch_experts_mt(const ExpertMaps &maps, const ExpertArgs &a_in, int num_sms, cudaStream_t st)
{
    static size_t configured = 0;
    static int blocks_per_sm = 0;
    ExpertArgs a = a_in;
    a.nstage = ring_stages(a.H, a.F, MT);
    const size_t smem = experts_smem_bytes_mt(a.H, a.F, MT, a.nstage);
    if (smem != configured) {
        if (cudaFuncSetAttribute(k_experts<MT, BPS, WB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return -1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, k_experts<MT, BPS, WB>, Cons<MT>::THREADS,
                                                          smem) != cudaSuccess ||
            blocks_per_sm < 1)
            return -1;
        configured = smem;
    }
    // every block must be resident: down units wait on gate/up units of others
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms * blocks_per_sm);
    cfg.blockDim = dim3(Cons<MT>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_experts<MT, BPS, WB>, maps, a) != cudaSuccess) return -1;
    count_launch();
    return 0;
}

template <int BPS, int WB>
static int launch_experts_bps(const ExpertMaps &maps, const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    // tiles hold at most min(T, GEMV_MT) tokens
    const int mt = a.n_tok < GEMV_MT ? a.n_tok : GEMV_MT;
    if (mt <= 1) return launch_experts_mt<1, BPS, WB>(maps, a, num_sms, st);
    if (mt <= 2) return launch_experts_mt<2, BPS, WB>(maps, a, num_sms, st);
    return launch_experts_mt<4, BPS, WB>(maps, a, num_sms, st);
}

int launch_experts(const ExpertMaps &maps, const ExpertArgs &a, int num_sms, cudaStream_t st)
{
    if (a.wbits == 8) {
        if (a.KC == 128) return launch_experts_bps<4, 8>(maps, a, num_sms, st);
        if (a.KC == 64) return launch_experts_bps<2, 8>(maps, a, num_sms, st);
        if (a.KC == 32) return launch_experts_bps<1, 8>(maps, a, num_sms, st);
        return -1;
    }
    if (a.KC == 128) return launch_experts_bps<8, 4>(maps, a, num_sms, st);
    if (a.KC == 64) return launch_experts_bps<4, 4>(maps, a, num_sms, st);
    if (a.KC == 16) return launch_experts_bps<1, 4>(maps, a, num_sms, st);
    return -1;
}

}  // namespace coli
