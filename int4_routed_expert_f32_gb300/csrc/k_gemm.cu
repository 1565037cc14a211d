// k_gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA-staged operands) for batches in which
// experts receive many tokens (prefill, large verify batches): the batch-union
// MoE of "Colibri: an AI engine running a 744B model in 25GB of RAM"
// (alphamatch.ai), section "Technical excellence", with the integer block dot
// products of "colibri: a pure-C inference engine ..." (discuss.pytorch.kr),
// section "Key features".
//
// Exactness.  The method multiplies int4 weights (-8..7) by int8 activations
// (-127..127) and sums each 32-element block in int32.  Both factors are exact
// in bf16, every product is exact, and a 32-term block sum (|sum| < 2^15) is
// exact in an F32 accumulator, so tcgen05.mma.kind::f16 on bf16 operands
// produces exactly the integers I_b.  (There is no kind::i8 on sm_103a.)  Each
// Q8_0 block gets its own TMEM accumulator (two K=16 MMAs), and the drain
// folds the blocks into F32 in ascending order, acc = fma(d_b, I_b, acc), the
// same operation sequence as the GEMV kernel and the CPU oracle, so the result
// is bit-identical to both.
//
// Tile.  M = 128 dispatch positions (rows of operand A: the gathered bf16
// codes of one expert's tokens), N = 256 weight rows (gate/up: 128 gate rows
// and the 128 matching up rows; down: 256 output rows), K = 64 per pipeline
// stage (two blocks).  The per-block exact fold makes every block a round
// trip between the MMA thread and the drain warps, and each round trip costs
// a roughly fixed number of cycles (MMA issue from one thread, commit, two
// mbarrier hand-offs) whatever N is; N = 256, the widest single-CTA MMA,
// gives each round trip the most work.  TMEM holds two such accumulators
// (2 x 256 columns): the MMAs of one block run while the other is drained.
// A drain thread owns one token row and 64 columns: 32 gate columns and the
// 32 up columns of the same hidden units (down: two groups of 32 output
// rows), so the per-(token, block) scale is one scalar, and SiLU(gate)*up and
// the requantisation of that Q8_0 block of h stay inside the thread.
//
// Warp roles (20 warps = 5 warpgroups, one CTA per SM, persistent over units):
//   0      TMA producer (activation tile + packed weight rows)
//   1      MMA issuer, owner of the TMEM allocation
//   2..3   weight converters: packed int4 -> bf16 in the 128-byte-swizzled
//          K-major layout the MMA reads
//   4..19  drain + epilogue; warp w reads TMEM lanes 32*(w%4).. and columns
//          32*((w-4)/4) .. and 128 + 32*((w-4)/4) .. of an accumulator.
//
// Element order inside each 8-element K chunk, for both operands:
// (k0, k2, k4, k6, k1, k3, k5, k7).  It is what splitting the packed bytes
// into low and high nibbles gives without shuffling; the gathered activations
// are written in the same order (one fixed permutation of K applied to both
// operands leaves every dot product unchanged).
#include <cuda.h>
#include <cuda_bf16.h>

#include "coli_common.cuh"
#include "coli_internal.h"
#include "tma.cuh"

namespace coli {

constexpr int GM = 128;                 // positions per tile (MMA M)
constexpr int GN = 256;                 // weight rows per tile (MMA N)
constexpr int GK = 64;                  // K per stage (two Q8_0 blocks)
constexpr int G_STAGES = 4;             // pipeline stages (int4 weights; int8 weights take 3)
constexpr int G_NACC = 2;               // TMEM accumulators (one per block in flight)
constexpr int A_BYTES = GM * GK * 2;    // 16 KB bf16, swizzled
constexpr int B_BYTES = GN * GK * 2;    // 32 KB bf16, swizzled

// Stages and packed-weight bytes per stage of each weight container: 8 KB of
// int4 nibbles or 16 KB of int8 codes (256 rows x 64 weights).
template <int WB> struct GemmCfg {
    static constexpr int STAGES = WB == 4 ? 4 : 3;
    static constexpr int RB = GK * WB / 8;          // packed bytes of a row per stage
    static constexpr int RAW_BYTES = GN * RB;
};
constexpr int G_CONV_WARPS = 2;
constexpr int G_DRAIN_WARP0 = 4;        // warps 0..3: producer, MMA, two converters
constexpr int G_DRAIN_WARPS = 16;       // 4 TMEM lane quarters x 4 column groups
constexpr int G_THREADS = 32 * (G_DRAIN_WARP0 + G_DRAIN_WARPS);
// Register split (setmaxnreg, per warpgroup): the control warpgroup gives
// registers to the four drain warpgroups (64 F32 accumulators per thread).
// The launch allocation must cover the sum; the launcher checks it against
// the compiled register count.
constexpr int G_REGS_CTRL = 64;
constexpr int G_REGS_DRAIN = 104;
constexpr int G_TMEM_COLS = G_NACC * GN;
constexpr uint64_t G_WAIT_NS = 2000000000ull;

static_assert(G_TMEM_COLS <= 512, "TMEM has 512 columns");
static_assert(32L * 4 * G_REGS_CTRL + 32L * G_DRAIN_WARPS * G_REGS_DRAIN <= 65536, "register split");

__device__ __forceinline__ uint64_t g_timer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded mbarrier wait that also gives up as soon as another warp aborted.
__device__ __forceinline__ bool g_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = g_timer();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (g_timer() - t0 > G_WAIT_NS) return false;
    }
}

// L2 policy of the weight copies.  A weight tile is read by every item of its
// expert (the shared expert has one item per 128 tokens) at about the same
// time; marking the copies evict-first lost those hits (1.5 times the
// algorithmic bytes of DRAM traffic per gate/up launch, against 1.02 with the
// normal policy).
__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Optional stage log.  Each block's region holds four sub-logs: 0 producer
// (code 11: stage issued), 1 reserved for the MMA issuer (which stays
// untraced: its loop bounds the tensor pipe), 2 first converter warp (14:
// stage landed, 15: stage converted), 3 first drain warp (16: block's
// accumulator ready, 17: block folded).  Entry i >= 1 of a sub-log is
// ((globaltimer << 8) | code, value), the timer's top bits dropped; entry 0
// receives the event count when the role finishes (the count lives in a
// register meanwhile, so logging adds no memory round trip).  Only stages
// [tr0, tr0 + TRACE_NS) of each block (and their blocks) are logged: a
// steady-state window after the first unit.
constexpr int TRACE_NS = 40;

__device__ __forceinline__ void gtrace(const GemmArgs &g, int role, int &n, int code, int value)
{
    if (n + 1 >= g.trace_cap / 4) return;
    unsigned long long *sub = g.trace + ((size_t)blockIdx.x * g.trace_cap + (size_t)role * (g.trace_cap / 4)) * 2;
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    ++n;
    sub[2 * n] = (t << 8) | (unsigned)code;
    sub[2 * n + 1] = (unsigned long long)value;
}

__device__ __forceinline__ void gtrace_close(const GemmArgs &g, int role, int n)
{
    if (!g.trace) return;
    g.trace[((size_t)blockIdx.x * g.trace_cap + (size_t)role * (g.trace_cap / 4)) * 2] = (unsigned long long)n;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: bf16 x bf16 -> F32, both operands K-major, M = GM, N = GN.
constexpr uint32_t UMMA_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GN >> 3) << 17) |
                                ((uint32_t)(GM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem, uint64_t da, uint64_t db, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem), "l"(da), "l"(db), "r"(UMMA_IDESC), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Eight int8 codes (natural order, little-endian in c) -> 16 bytes of bf16 in
// chunk order (k0, k2, k4, k6, k1, k3, k5, k7).  |code| <= 127 is exact in bf16.
__device__ __forceinline__ uint4 codes_to_bf16_chunk(uint2 c)
{
    const uint32_t lo = __byte_perm(c.x, c.y, 0x6420), hi = __byte_perm(c.x, c.y, 0x7531);
    const uint32_t src[2] = {lo, hi};
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float a = (float)(int8_t)(src[h] >> (16 * p));
            const float b = (float)(int8_t)(src[h] >> (16 * p + 8));
            w[2 * h + p] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 4 bytes of packed nibbles (8 weights; element 2i in the low nibble of byte
// i) -> 16 bytes of bf16 (nibble - 8) in chunk order.  The bf16 pattern 0x43nn
// (nn < 16) is 128 + nn; subtracting 136 leaves nn - 8 exactly.
__device__ __forceinline__ uint4 nibbles_to_bf16_chunk(uint32_t w)
{
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t C = 0x43434343u;
    uint32_t o[4] = {__byte_perm(lo, C, 0x4140), __byte_perm(lo, C, 0x4342), __byte_perm(hi, C, 0x4140),
                     __byte_perm(hi, C, 0x4342)};
    const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&o[i]);
        v = __hsub2(v, bias);
        o[i] = *reinterpret_cast<uint32_t *>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// Gather: the bf16 chunk-ordered codes of every used dispatch position (the A
// operand of the gate/up GEMM).  Positions [offsets[E], P) hold no pair (an
// invalid expert index) and are skipped.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gather_x(const int8_t *__restrict__ qx,
                                                  const int32_t *__restrict__ pos_token,
                                                  const int32_t *__restrict__ offsets, int E, int P, int R,
                                                  int T, int H, uint16_t *__restrict__ xg, int *status)
{
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;   // one 8-element chunk
    const int per = H / 8;
    if (i >= (long)R * per) return;
    const int pos = (int)(i / per), c = (int)(i - (long)pos * per);
    if (pos < P && pos >= offsets[E]) return;
    const int tok = pos_token[pos];
    if (tok < 0 || tok >= T) {
        set_status(status, ST_BAD_INDEX);
        return;
    }
    const uint2 codes = *reinterpret_cast<const uint2 *>(qx + (size_t)tok * H + (size_t)c * 8);
    reinterpret_cast<uint4 *>(xg + (size_t)pos * H)[c] = codes_to_bf16_chunk(codes);
}

// GEMM work items: each expert's dispatch positions in tiles of GM, the shared
// expert (rows P .. P+T-1) first, then routed experts in ascending id.  One
// block of 256 threads (E <= 256): thread e counts expert e's tiles, a block
// scan gives its first item, and every thread writes its own items.
__global__ void __launch_bounds__(256) k_gemm_items(const int32_t *__restrict__ counts,
                                                    const int32_t *__restrict__ offsets, int E, int T, int P,
                                                    int32_t *item_expert, int32_t *item_pos0, int32_t *item_m,
                                                    int32_t *n_items)
{
    __shared__ int s_warp[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int shared_items = (T + GM - 1) / GM;
    for (int q = tid; q < shared_items; q += blockDim.x) {
        item_expert[q] = E;
        item_pos0[q] = P + q * GM;
        item_m[q] = min(GM, T - q * GM);
    }
    const int cnt = tid < E ? counts[tid] : 0;
    const int ni = (cnt + GM - 1) / GM;
    // inclusive scan of the tile counts: within the warp, then over the warps
    int inc = ni;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int v = s_warp[w];
        before += (w < warp) ? v : 0;
        total += v;
    }
    const int first = shared_items + before + inc - ni;
    if (tid < E) {
        const int off = offsets[tid];
        for (int q = 0; q < ni; ++q) {
            item_expert[first + q] = tid;
            item_pos0[first + q] = off + q * GM;
            item_m[first + q] = min(GM, cnt - q * GM);
        }
    }
    if (tid == 0) *n_items = shared_items + total;
}

// Combine: out[t] = y[shared row of t], then + w_r * y[pair (t, r)] for the
// ranks r in order, one fused multiply-add each (the method's weighted sum of
// the shared expert and the k routed experts); with `res`, the residual of a
// stacked decoder is added last: out = res + that sum.
__global__ void __launch_bounds__(256) k_combine(const float *__restrict__ y, const int32_t *__restrict__ inv,
                                                 const float *__restrict__ wts, int T, int k, int P, int H,
                                                 const float *__restrict__ res, float *__restrict__ out)
{
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;   // 4 columns
    const int per = H / 4;
    if (i >= (long)T * per) return;
    const int t = (int)(i / per), c = (int)(i - (long)t * per);
    float4 o = reinterpret_cast<const float4 *>(y + (size_t)(P + t) * H)[c];
    for (int r = 0; r < k; ++r) {
        const int pos = inv[(size_t)t * k + r];
        if (pos < 0 || pos >= P) continue;
        const float w = wts[(size_t)t * k + r];
        const float4 v = reinterpret_cast<const float4 *>(y + (size_t)pos * H)[c];
        o.x = __fmaf_rn(w, v.x, o.x);
        o.y = __fmaf_rn(w, v.y, o.y);
        o.z = __fmaf_rn(w, v.z, o.z);
        o.w = __fmaf_rn(w, v.w, o.w);
    }
    if (res) {
        const float4 r = reinterpret_cast<const float4 *>(res + (size_t)t * H)[c];
        o.x = __fadd_rn(r.x, o.x);
        o.y = __fadd_rn(r.y, o.y);
        o.z = __fadd_rn(r.z, o.z);
        o.w = __fadd_rn(r.w, o.w);
    }
    reinterpret_cast<float4 *>(out + (size_t)t * H)[c] = o;
}

struct GemmSmem {
    alignas(8) uint64_t full[G_STAGES];      // activation tile + packed weights landed (TMA)
    alignas(8) uint64_t conv[G_STAGES];      // weights converted to bf16
    alignas(8) uint64_t empty[G_STAGES];     // the stage's MMAs completed
    alignas(8) uint64_t tfull[G_NACC];       // a block's accumulator is ready
    alignas(8) uint64_t tempty[G_NACC];      // a block's accumulator was read
    uint32_t tmem_base;
    int abort;
};

template <int WB>
static size_t gemm_smem_bytes_w()
{
    return 1024 + (size_t)GemmCfg<WB>::STAGES * (A_BYTES + B_BYTES + GemmCfg<WB>::RAW_BYTES) + sizeof(GemmSmem);
}

size_t gemm_smem_bytes() { return gemm_smem_bytes_w<4>(); }

// GATEUP: A = gathered x codes (K = H), B = gate/up rows; epilogue SiLU*up and
// Q8_0 of h.  Otherwise A = h codes (K = F), B = down rows; epilogue y.
// WB: weight container, 4 (packed int4) or 8 (int8 codes).
template <bool GATEUP, int WB>
__global__ void __launch_bounds__(G_THREADS, 1)
k_gemm(const __grid_constant__ GemmMaps maps, const GemmArgs g)
{
    constexpr int G_STAGES = GemmCfg<WB>::STAGES;
    constexpr int RB = GemmCfg<WB>::RB;
    constexpr int RAW_BYTES = GemmCfg<WB>::RAW_BYTES;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *sA = smem;                                   // [G_STAGES][A_BYTES]
    unsigned char *sB = sA + G_STAGES * A_BYTES;                // [G_STAGES][B_BYTES]
    unsigned char *sRaw = sB + G_STAGES * B_BYTES;              // [G_STAGES][RAW_BYTES]
    GemmSmem &S = *reinterpret_cast<GemmSmem *>(sRaw + G_STAGES * RAW_BYTES);
    volatile int *abort = &S.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = g.H, F = g.F;
    const int K = GATEUP ? H : F;
    const int nst = K / GK;                         // stages per unit
    const int nb = K / 32;                          // blocks per unit
    // weight tiles per item: F/128 gate/up tiles; ceil(H/256) down tiles (the
    // last one half past the matrix when H is an odd multiple of 128: the TMA
    // box reads zeros there and the drain stores nothing for those rows)
    const int per_item = GATEUP ? F / (GN / 2) : (H + GN - 1) / GN;
    const int n_units = *g.n_items * per_item;
    const int tr0 = nst + 8;                       // first traced stage
    const bool tr = g.trace != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.conv[s], G_CONV_WARPS);
            mbar_init(&S.empty[s], 1);
        }
        for (int b = 0; b < G_NACC; ++b) {
            mbar_init(&S.tfull[b], 1);
            mbar_init(&S.tempty[b], G_DRAIN_WARPS);   // one arrival per drain warp
        }
        S.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&maps.act);
        prefetch_tmap(&maps.w);
        prefetch_tmap(&maps.sw);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&S.tmem_base)), "r"(G_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    // Role dispatch.  Each warpgroup changes its register share inside its
    // own branch, so that the compiler applies the drain's larger budget to
    // the drain code only.
    if (warp < G_DRAIN_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(G_REGS_CTRL));
    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            int ntr = 0;
            int sc = 0;   // stages issued
            for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
                const int item = u / per_item, j = u - item * per_item;
                const int e = g.item_expert[item], pos0 = g.item_pos0[item];
                const bool shared = (e == g.E);
                const void *wmap = shared ? (const void *)&maps.sw : (const void *)&maps.w;
                const int z = shared ? 0 : (g.slot_of ? g.slot_of[e] : e);
                for (int s = 0; s < nst; ++s, ++sc) {
                    const int slot = sc % G_STAGES;
                    const int rnd = sc / G_STAGES;
                    if (rnd > 0 && !g_wait(&S.empty[slot], (uint32_t)((rnd - 1) & 1), abort)) {
                        if (!*abort) set_status(g.status, ST_TIMEOUT);
                        *abort = 1;
                        break;
                    }
                    if (tr && sc >= tr0 && sc < tr0 + TRACE_NS) gtrace(g, 0, ntr, 11, sc);
                    mbar_arrive_expect_tx(&S.full[slot], A_BYTES + RAW_BYTES);
                    tma_load_2d(sA + slot * A_BYTES, &maps.act, s * GK, pos0, &S.full[slot]);
                    unsigned char *raw = sRaw + slot * RAW_BYTES;
                    if (GATEUP) {
                        // 128 gate rows, then the 128 matching up rows (RB bytes each)
                        tma_load_3d(raw, wmap, s * RB, (GN / 2) * j, z, &S.full[slot], pol);
                        tma_load_3d(raw + (GN / 2) * RB, wmap, s * RB, F + (GN / 2) * j, z, &S.full[slot], pol);
                    } else {
                        tma_load_3d(raw, wmap, s * RB, GN * j, z, &S.full[slot], pol);
                    }
                }
            }
            gtrace_close(g, 0, ntr);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        // One thread issues every MMA of the CTA.  Per stage: one wait for the
        // converted operands (which implies the TMA data), then per block one
        // wait for its accumulator to be drained, a fence, two K = 16 MMAs and
        // a commit; a last commit frees the stage.
        if (lane == 0) {
            const int my_units =
                (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
            const int total = my_units * nst;
            const uint64_t dA = umma_desc(smem_u32(sA)), dB = umma_desc(smem_u32(sB));
            int slot = 0;
            uint32_t phase = 0;
            bool failed = false;
            for (int sc = 0; sc < total && !failed; ++sc) {
                if (!g_wait(&S.conv[slot], phase, abort)) {
                    failed = true;
                    break;
                }
                // descriptor start addresses advance in 16-byte units: +2 per 32 bytes of K
                const uint64_t da = dA + (uint64_t)(slot * (A_BYTES >> 4));
                const uint64_t db = dB + (uint64_t)(slot * (B_BYTES >> 4));
#pragma unroll
                for (int h = 0; h < G_NACC; ++h) {
                    // block 2 sc + h goes to accumulator h, whose previous block was drained
                    if (sc > 0 && !g_wait(&S.tempty[h], (uint32_t)((sc - 1) & 1), abort)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(h * GN);
                    umma_bf16(d, da + 4 * h, db + 4 * h, 0u);
                    umma_bf16(d, da + 4 * h + 2, db + 4 * h + 2, 1u);
                    umma_commit(&S.tfull[h]);
                }
                if (failed) break;
                umma_commit(&S.empty[slot]);    // the stage's operands may be overwritten
                if (++slot == G_STAGES) {
                    slot = 0;
                    phase ^= 1;
                }
            }
            if (failed) {
                if (!*abort) set_status(g.status, ST_TIMEOUT);
                *abort = 1;
            } else if (total > 0) {
                // the last commit to `empty` must land before the CTA exits
                const int last = total - 1;
                if (!g_wait(&S.empty[last % G_STAGES], (uint32_t)((last / G_STAGES) & 1), abort)) {
                    set_status(g.status, ST_TIMEOUT);
                    *abort = 1;
                }
            }
        }
    } else {
        // ------------------------------ converters ------------------------------
        // packed weights [GN rows][RB bytes] -> bf16 [GN][GK] in the swizzled layout
        const int ct = threadIdx.x - 32 * 2;        // 0 .. 63
        constexpr int PIECES = GN * 2;              // (row, block) pieces of RB/2 packed bytes per stage
        constexpr int PER = PIECES / (32 * G_CONV_WARPS);
        constexpr int BATCH = WB == 4 ? 4 : 2;      // packed loads in flight per thread
        static_assert(PER % BATCH == 0, "converter batches");
        int sc = 0;
        int ntr = 0;
        for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
            for (int s = 0; s < nst; ++s, ++sc) {
                const int slot = sc % G_STAGES;
                const uint32_t par = (uint32_t)((sc / G_STAGES) & 1);
                const bool ok = __all_sync(FULL, g_wait(&S.full[slot], par, abort));
                if (!ok) {
                    if (lane == 0) {
                        if (!*abort) set_status(g.status, ST_TIMEOUT);
                        *abort = 1;
                    }
                    break;
                }
                const bool trc = tr && warp == 2 && lane == 0 && sc >= tr0 && sc < tr0 + TRACE_NS;
                if (trc) gtrace(g, 2, ntr, 14, sc);
                const unsigned char *raw = sRaw + slot * RAW_BYTES;
                unsigned char *bt = sB + slot * B_BYTES;
#pragma unroll 1
                for (int p0 = 0; p0 < PER; p0 += BATCH) {
                    // piece (row n, block blk) is RB/2 bytes at n * RB + blk * RB / 2 = piece * RB / 2
                    uint4 w[BATCH][WB / 4];
#pragma unroll
                    for (int i = 0; i < BATCH; ++i)
#pragma unroll
                        for (int h = 0; h < WB / 4; ++h)
                            w[i][h] = *reinterpret_cast<const uint4 *>(raw + (size_t)(ct + 64 * (p0 + i)) * (RB / 2) +
                                                                        16 * h);
#pragma unroll
                    for (int i = 0; i < BATCH; ++i) {
                        const int piece = ct + 64 * (p0 + i);
                        const int n = piece >> 1, blk = piece & 1;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int c = blk * 4 + q;   // 8-element chunk along K
                            uint4 o;
                            if (WB == 4) {
                                const uint32_t wv[4] = {w[i][0].x, w[i][0].y, w[i][0].z, w[i][0].w};
                                o = nibbles_to_bf16_chunk(wv[q]);
                            } else {
                                const uint4 &hv = w[i][(WB / 4 - 1) & (q >> 1)];
                                o = codes_to_bf16_chunk((q & 1) ? make_uint2(hv.z, hv.w) : make_uint2(hv.x, hv.y));
                            }
                            *reinterpret_cast<uint4 *>(bt + n * 128 + ((c ^ (n & 7)) << 4)) = o;
                        }
                    }
                }
                fence_proxy_async_shared();   // generic-proxy writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.conv[slot]);
                if (trc) gtrace(g, 2, ntr, 15, sc);
            }
        }
        if (warp == 2 && lane == 0) gtrace_close(g, 2, ntr);
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(G_REGS_DRAIN));
        // ------------------------------ drain / epilogue ------------------------------
        // Every drain warp walks the same units and blocks (also after an
        // abort, without touching data) so that every accumulator hand-off
        // sees all sixteen arrivals.
        const int dw = warp - G_DRAIN_WARP0;         // 0 .. 15
        const int quad = warp & 3;                   // TMEM lanes 32*quad ..
        const int cq = dw >> 2;                      // columns 32*cq .. and 128 + 32*cq ..
        const int row = 32 * quad + lane;            // position row of the tile
        int bc = 0;
        int ntr = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            const int item = u / per_item, j = u - item * per_item;
            const int e = g.item_expert[item], pos0 = g.item_pos0[item], m = g.item_m[item];
            const bool active = 32 * quad < m;       // warp-uniform: any valid row in this quad
            const bool valid = row < m;
            const int pos = pos0 + (valid ? row : 0);
            const float *dsc;
            if (GATEUP) {
                int tok = valid ? g.pos_token[pos] : 0;
                if (tok < 0 || tok >= g.T) tok = 0;   // flagged by the gather kernel
                dsc = g.dx + (size_t)tok * (H / 32);
            } else {
                dsc = g.dh + (size_t)pos * (F / 32);
            }
            // acc[0..15]: columns 32cq .. +31, acc[16..31]: columns 128 + 32cq .. +31
            float2 acc[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) acc[c] = make_float2(0.0f, 0.0f);
            // block scales in groups of 4 (nb % 4 == 0), the next group loaded
            // while this one is folded
            const float4 zero4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const float4 *dsc4 = reinterpret_cast<const float4 *>(dsc);
            float4 dnext = valid ? __ldg(dsc4) : zero4;
            for (int b4 = 0; b4 < nb; b4 += 4) {
                const float4 dcur = dnext;
                if (valid && b4 + 4 < nb) dnext = __ldg(dsc4 + (b4 >> 2) + 1);
#pragma unroll
                for (int bi = 0; bi < 4; ++bi, ++bc) {
                    const float db = bi == 0 ? dcur.x : bi == 1 ? dcur.y : bi == 2 ? dcur.z : dcur.w;
                    const int a = bc & 1;
                    const uint32_t par = (uint32_t)((bc >> 1) & 1);
                    const bool ok = !*abort && __all_sync(FULL, g_wait(&S.tfull[a], par, abort));
                    const bool trd = tr && dw == 0 && lane == 0 && bc >= 2 * tr0 && bc < 2 * (tr0 + TRACE_NS);
                    if (trd) gtrace(g, 3, ntr, 16, bc);
                    if (ok) {
                        tc_fence_after();
                        if (active) {
                            const uint32_t base =
                                tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(a * GN + 32 * cq);
                            const float2 dd = make_float2(db, db);
#pragma unroll
                            for (int hq = 0; hq < 4; ++hq) {
                                // 16 columns: half hq/2 (+128 columns), quarter hq%2
                                float v[16];
                                tmem_ld16(base + (uint32_t)(128 * (hq >> 1) + 16 * (hq & 1)), v);
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    acc[8 * hq + c] =
                                        __ffma2_rn(dd, make_float2(v[2 * c], v[2 * c + 1]), acc[8 * hq + c]);
                            }
                        }
                        tc_fence_before();
                    } else if (lane == 0) {
                        if (!*abort) set_status(g.status, ST_TIMEOUT);
                        *abort = 1;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.tempty[a]);
                    if (trd) gtrace(g, 3, ntr, 17, bc);
                }
            }
            const bool live = !*abort;
            // ---- epilogue ----
            const float *ers = (e == g.E) ? g.shared_rs
                                          : g.expert_rs + (size_t)(g.slot_of ? g.slot_of[e] : e) * (2 * F + H);
            if (GATEUP) {
                if (live && valid) {
                    // hidden units 128j + 32cq .. +31 of this token: one Q8_0 block of h
                    const int col0 = (GN / 2) * j + 32 * cq;
                    const float *sg = ers + col0, *su = ers + F + col0;
                    float h[32];
                    float amax = 0.0f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float gv = (c & 1) ? acc[c >> 1].y : acc[c >> 1].x;
                        const float uv = (c & 1) ? acc[16 + (c >> 1)].y : acc[16 + (c >> 1)].x;
                        const float gg = __fmul_rn(sg[c], gv);
                        const float uu = __fmul_rn(su[c], uv);
                        h[c] = __fmul_rn(__fmul_rn(gg, own_sigmoid(gg)), uu);
                        amax = fmaxf(amax, fabsf(h[c]));
                    }
                    const float dq = __fdiv_rn(amax, 127.0f);
                    const float id = (dq != 0.0f) ? __fdiv_rn(1.0f, dq) : 0.0f;
                    uint32_t qw[8];
#pragma unroll
                    for (int w4 = 0; w4 < 8; ++w4) {
                        uint32_t word = 0;
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) {
                            int q = __float2int_rn(__fmul_rn(h[4 * w4 + bb], id));
                            q = max(-127, min(127, q));
                            word |= ((uint32_t)q & 0xFFu) << (8 * bb);
                        }
                        qw[w4] = word;
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(g.qh + (size_t)pos * F + col0);
                    dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                    dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
                    g.dh[(size_t)pos * (F / 32) + col0 / 32] = dq;
                    uint4 *bdst = reinterpret_cast<uint4 *>(g.qhb + (size_t)pos * F + col0);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        bdst[c8] = codes_to_bf16_chunk(make_uint2(qw[2 * c8], qw[2 * c8 + 1]));
                    if (g.h_dbg) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) g.h_dbg[(size_t)pos * F + col0 + c] = h[c];
                    }
                }
            } else if (live && valid) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int col0 = GN * j + 128 * hh + 32 * cq;
                    if (GN * j + 128 * hh < H) {          // H % 128 == 0: the half is whole or absent
                        float4 *yr = reinterpret_cast<float4 *>(g.y + (size_t)pos * H + col0);
                        const float *sd = ers + 2 * F + col0;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            float4 o;
                            o.x = __fmul_rn(sd[4 * c], acc[16 * hh + 2 * c].x);
                            o.y = __fmul_rn(sd[4 * c + 1], acc[16 * hh + 2 * c].y);
                            o.z = __fmul_rn(sd[4 * c + 2], acc[16 * hh + 2 * c + 1].x);
                            o.w = __fmul_rn(sd[4 * c + 3], acc[16 * hh + 2 * c + 1].y);
                            yr[c] = o;
                        }
                    }
                }
            }
        }
        if (dw == 0 && lane == 0) gtrace_close(g, 3, ntr);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G_TMEM_COLS));
    }
}

int launch_gather_x(const int8_t *qx, const int32_t *pos_token, const int32_t *offsets, int E, int P, int R,
                    int T, int H, uint16_t *xg, int *status, cudaStream_t st)
{
    const long n = (long)R * (H / 8);
    if (n == 0) return 0;
    k_gather_x<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(qx, pos_token, offsets, E, P, R, T, H, xg, status);
    count_launch();
    return 0;
}

int launch_gemm_items(const int32_t *counts, const int32_t *offsets, int E, int T, int P, int32_t *item_expert,
                      int32_t *item_pos0, int32_t *item_m, int32_t *n_items, cudaStream_t st)
{
    k_gemm_items<<<1, 256, 0, st>>>(counts, offsets, E, T, P, item_expert, item_pos0, item_m, n_items);
    count_launch();
    return 0;
}

int launch_combine(const float *y, const int32_t *inv, const float *wts, int T, int k, int P, int H,
                   const float *res, float *out, cudaStream_t st)
{
    const long n = (long)T * (H / 4);
    if (n == 0) return 0;
    k_combine<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, inv, wts, T, k, P, H, res, out);
    count_launch();
    return 0;
}

int max_gemm_items(int T, int k, int E)
{
    const long P = (long)T * k;
    return (int)(P / GM + (P < E ? P : E) + 1 + (T + GM - 1) / GM);
}

int gemm_tile_rows() { return GM; }

template <bool GATEUP, int WB>
static int launch_gemm_t(const GemmMaps &maps, const GemmArgs &g, int num_sms, cudaStream_t st)
{
    static int configured_device = -1;
    const size_t smem = gemm_smem_bytes_w<WB>();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (configured_device != dev) {
        // setmaxnreg.inc waits until enough registers are free: the warpgroups'
        // shares after the split must fit in what the CTA is launched with
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, k_gemm<GATEUP, WB>) != cudaSuccess) return -1;
        const long have = (long)fa.numRegs * G_THREADS;
        const long need = 32L * G_DRAIN_WARP0 * G_REGS_CTRL + 32L * G_DRAIN_WARPS * G_REGS_DRAIN;
        if (fa.numRegs < G_REGS_CTRL || fa.numRegs > G_REGS_DRAIN || need > have) return -1;
        if (cudaFuncSetAttribute(k_gemm<GATEUP, WB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return -1;
        configured_device = dev;
    }
    k_gemm<GATEUP, WB><<<num_sms, G_THREADS, smem, st>>>(maps, g);
    count_launch();
    return 0;
}

int launch_gemm(bool gateup, int wbits, const GemmMaps &maps, const GemmArgs &g, int num_sms, cudaStream_t st)
{
    if (wbits == 8)
        return gateup ? launch_gemm_t<true, 8>(maps, g, num_sms, st) : launch_gemm_t<false, 8>(maps, g, num_sms, st);
    return gateup ? launch_gemm_t<true, 4>(maps, g, num_sms, st) : launch_gemm_t<false, 4>(maps, g, num_sms, st);
}

}  // namespace coli
