// coli_moe.cu -- the C ABI (include/coli_moe.h): argument checks, the
// library-owned workspace, and the launch sequence of one MoE layer forward.
//
// Forward sequence on the caller's stream (no host synchronisation):
//   routing, T <= 8: one launch (k_route_small) doing Q8_0 of x, the router
//   logits in the fixed F32 order, sigmoid/top-k/renormalisation, the stable
//   token->expert dispatch and the tile list;
//   routing, T > 8: k_q8_0, k_router_logits, k_topk, k_dispatch;
//   experts, streaming path (decode batches): one persistent launch
//   (k_experts): gate/up + SiLU*up + Q8_0 of h, down, and the gate-weighted
//   combine with the shared expert;
//   experts, grouped tensor-core path (prefill batches): k_gather_x (bf16
//   codes by dispatch position), k_gemm_items (tiles of 128 positions per
//   expert), k_gemm<gate/up> (+ SiLU*up + Q8_0 of h), k_gemm<down>, k_combine.
#include <cstdio>
#include <cstring>
#include <utility>
#include <vector>

#include "../../include/coli_moe.h"
#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

static long long g_launches = 0;
void count_launch() { ++g_launches; }

struct Workspace {
    void *base = nullptr;
    size_t bytes = 0;
    int8_t *qx = nullptr;
    float *dx = nullptr;
    float *logits = nullptr;
    float *sig = nullptr, *key = nullptr;
    int32_t *idx = nullptr;
    float *wts = nullptr;
    int32_t *counts = nullptr, *offsets = nullptr, *perm = nullptr, *inv = nullptr;
    int32_t *pos_token = nullptr;
    int32_t *tile_expert = nullptr, *tile_pos0 = nullptr, *tile_m = nullptr, *n_tiles = nullptr;
    int *sync = nullptr;            // g_done[max tiles] | w_done[H/64] | work counter
    int n_sync = 0;
    int *route_counter = nullptr;
    int8_t *qh = nullptr;
    float *dh = nullptr;
    float *y = nullptr;
    float *x_io = nullptr, *out_io = nullptr;
    float *xn = nullptr;             // [T][H] normalised input of a stacked layer
    int *status = nullptr;
    // grouped tensor-core path
    uint16_t *xg = nullptr;          // [R'][H] bf16 codes of x by dispatch position
    uint16_t *qhb = nullptr;         // [R'][F] bf16 codes of h by dispatch position
    int32_t *item_expert = nullptr, *item_pos0 = nullptr, *item_m = nullptr, *n_items = nullptr;
    int rows_alloc = 0;              // R' = max(P + T, 128) rows of xg and qhb
    // guard regions: from each piece's end to the next piece (at least
    // WS_GUARD bytes), and WS_GUARD bytes before the first piece, filled with
    // WS_GUARD_BYTE at configure; a write past a piece's end lands in one
    std::vector<std::pair<size_t, size_t>> guards;   // (offset, bytes)
};
constexpr size_t WS_GUARD = 256;
constexpr unsigned char WS_GUARD_BYTE = 0xA5;

struct State {
    bool configured = false;
    coli_moe_shape s{};
    int device = -1;
    int num_sms = 0;
    Workspace ws;
    int path = COLI_PATH_AUTO;
    int gemm_min_tokens = 0;
    bool timing = false;
    std::vector<cudaEvent_t> ev_pool;  // pairs (start, stop)
    int ev_used = 0;
    int max_tiles = 0;
    unsigned long long *trace = nullptr;   // expert-kernel event log (device)
    int trace_cap = 0;
    int trace_blocks = 0;
    // tensor maps of the last weights seen (re-encoded when a pointer changes)
    ExpertMaps maps{};
    const void *maps_key[2] = {nullptr, nullptr};
    int maps_wbits = 0;
    int maps_extent = 0;
    bool maps_valid = false;
    int wbits = 4;                   // weight container of later forwards (coli_moe_set_weight_bits)
    // grouped-GEMM maps: activations (fixed workspace buffers, encoded at
    // configure) and weights (re-encoded when a pointer, the weight
    // container or the weight array's extent changes)
    CUtensorMap act_x{}, act_h{};
    GemmMaps gemm_gu{}, gemm_dn{};
    const void *gemm_key[2] = {nullptr, nullptr};
    int gemm_wbits = 0;
    int gemm_extent = 0;
    bool gemm_valid = false;
};

static State g;

// Host-memory expert tier: routed experts live in host memory; an LRU cache
// of them lives in a pool of HBM slots (coli_moe_tier_*).
struct Tier {
    int n_slots = 0;
    int E = 0;
    int wbits = 4;
    size_t stride = 0;               // bytes of one expert's weights
    size_t rs_len = 0;               // row scales of one expert (2F + H)
    uint8_t *pool_w = nullptr;       // device [n_slots][stride]
    float *pool_rs = nullptr;        // device [n_slots][rs_len]
    int32_t *slot_dev = nullptr;     // device [E]: slot of each expert (valid for the forward's experts)
    int32_t *slot_host = nullptr;    // pinned [E]
    int32_t *idx_host = nullptr;     // pinned [max_tok * k]
    std::vector<int> slot_of;        // [E]: -1 when not resident
    std::vector<int> expert_in;      // [n_slots]: -1 when empty
    std::vector<long long> stamp;    // [n_slots]: last forward that used the slot (LRU)
    long long clock = 0, hits = 0, misses = 0, bytes = 0;
};
static Tier g_tier;

static void tier_free()
{
    if (g_tier.pool_w) cudaFree(g_tier.pool_w);
    if (g_tier.pool_rs) cudaFree(g_tier.pool_rs);
    if (g_tier.slot_dev) cudaFree(g_tier.slot_dev);
    if (g_tier.slot_host) cudaFreeHost(g_tier.slot_host);
    if (g_tier.idx_host) cudaFreeHost(g_tier.idx_host);
    g_tier = Tier{};
}

// Test-only failure injection (coli_moe_dbg_inject): host-side counters, so
// that nothing ever faults or hangs the GPU.
struct Inject {
    int alloc_fail = 0;          // workspace allocations that fail (no cudaMalloc call)
    int launch_fail_at = 0;      // the n-th launch from now reports failure (0: off)
    long long wait_us = 0;       // next streaming forward: unreachable gate/up wait, bound in us
};
static Inject g_inj;

// True when the injected launch failure is due now (the launch is skipped).
static bool inject_launch_failure()
{
    if (g_inj.launch_fail_at <= 0) return false;
    return --g_inj.launch_fail_at == 0;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int cuda_fail(cudaError_t e)
{
    (void)cudaGetLastError();
    (void)e;
    return COLI_E_CUDA;
}

#define CUDA_OK(call)                                  \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_);   \
    } while (0)

#define LAUNCH_OK(call)                                                        \
    do {                                                                       \
        if (inject_launch_failure()) return cuda_fail(cudaErrorLaunchFailure); \
        if ((call) != 0) return cuda_fail(cudaErrorUnknown);                   \
        cudaError_t e_ = cudaGetLastError();                                   \
        if (e_ != cudaSuccess) return cuda_fail(e_);                           \
    } while (0)

static void free_workspace()
{
    if (g.ws.base) cudaFree(g.ws.base);
    g.ws = Workspace{};
    for (cudaEvent_t e : g.ev_pool) cudaEventDestroy(e);
    g.ev_pool.clear();
    g.ev_used = 0;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ---- TMA tensor maps of the expert weights --------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// Bytes of a weight row per TMA box of the streaming kernel: the widest of
// 128 (128-byte swizzled boxes), 64, 32 and 16 that divides both row lengths
// in bytes (H * wbits / 8 and F * wbits / 8; H % 128 == 0 and F % 32 == 0).
// The kernel is instantiated for 128, 64 and 16 with int4 weights (F / 2 is a
// multiple of 16, and of 32 only when it is one of 64) and for 128, 64 and 32
// with int8 weights.
static int stage_kc(int H, int F, int wbits)
{
    const int rh = H * wbits / 8, rf = F * wbits / 8;
    if (rh % 128 == 0 && rf % 128 == 0) return 128;
    if (rf % 64 == 0) return 64;
    return wbits == 8 ? 32 : 16;
}

// The grouped GEMM's tiles need F % 128 == 0 (gate/up tiles of 128 hidden
// units; the down GEMM's K = F in stages of 64).
static bool gemm_shape_ok(int F) { return F % 128 == 0; }

// rows of `row_bytes` bytes, `n_exp` experts `exp_stride` bytes apart; box =
// kc bytes x box_rows rows of one expert
static bool encode_rows(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows,
                        uint64_t n_exp, uint64_t exp_stride, uint32_t box_rows, uint32_t kc)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {row_bytes, rows, n_exp};
    cuuint64_t strides[2] = {row_bytes, exp_stride};
    cuuint32_t box[3] = {kc, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    kc == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Maps for routed experts at `ew4` ([E][3FH/2]) and the shared expert at `sw4`.
static bool expert_maps(const uint8_t *ew4, int E, const uint8_t *sw4, ExpertMaps *out)
{
    if (g.maps_valid && g.maps_key[0] == ew4 && g.maps_key[1] == sw4 && g.maps_wbits == g.wbits &&
        g.maps_extent == E) {
        *out = g.maps;
        return true;
    }
    const uint64_t H = g.s.hidden, F = g.s.ffn, wb = (uint64_t)g.wbits;
    const uint64_t rh = H * wb / 8, rf = F * wb / 8, stride = 3 * F * H * wb / 8;
    const uint32_t kc = (uint32_t)stage_kc((int)H, (int)F, g.wbits);
    ExpertMaps m;
    bool ok = encode_rows(&m.gu, ew4, rh, 2 * F, (uint64_t)E, stride, 32, kc) &&
              encode_rows(&m.dn, ew4 + 2 * F * rh, rf, H, (uint64_t)E, stride, 64, kc) &&
              encode_rows(&m.sgu, sw4, rh, 2 * F, 1, stride, 32, kc) &&
              encode_rows(&m.sdn, sw4 + 2 * F * rh, rf, H, 1, stride, 64, kc);
    if (!ok) return false;
    g.maps = m;
    g.maps_key[0] = ew4;
    g.maps_key[1] = sw4;
    g.maps_wbits = g.wbits;
    g.maps_extent = E;
    g.maps_valid = true;
    *out = m;
    return true;
}

// 2-D map over bf16 codes [rows][K] with 128-byte swizzle, box 64 x 128.
static bool encode_act(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Weight maps of the grouped GEMM: the packed bytes of 64 weights of a row
// per stage (32 for int4, 64 for int8), 128 rows per box for gate/up (two
// boxes: gate rows, then the matching up rows), 256 rows for down (rows past
// the matrix read as zeros).  `E` is the extent of the routed-weight array.
static bool gemm_weight_maps(const uint8_t *ew4, int E, const uint8_t *sw4)
{
    if (g.gemm_valid && g.gemm_key[0] == ew4 && g.gemm_key[1] == sw4 && g.gemm_wbits == g.wbits &&
        g.gemm_extent == E)
        return true;
    const uint64_t H = g.s.hidden, F = g.s.ffn, wb = (uint64_t)g.wbits;
    const uint64_t rh = H * wb / 8, rf = F * wb / 8, stride = 3 * F * H * wb / 8;
    const uint32_t rb = (uint32_t)(64 * wb / 8);
    GemmMaps gu{}, dn{};
    bool ok = encode_rows(&gu.w, ew4, rh, 2 * F, (uint64_t)E, stride, 128, rb) &&
              encode_rows(&gu.sw, sw4, rh, 2 * F, 1, stride, 128, rb) &&
              encode_rows(&dn.w, ew4 + 2 * F * rh, rf, H, (uint64_t)E, stride, 256, rb) &&
              encode_rows(&dn.sw, sw4 + 2 * F * rh, rf, H, 1, stride, 256, rb);
    if (!ok) {
        g.gemm_valid = false;
        return false;
    }
    gu.act = g.act_x;
    dn.act = g.act_h;
    g.gemm_gu = gu;
    g.gemm_dn = dn;
    g.gemm_key[0] = ew4;
    g.gemm_key[1] = sw4;
    g.gemm_wbits = g.wbits;
    g.gemm_extent = E;
    g.gemm_valid = true;
    return true;
}

static int check_shape(const coli_moe_shape *s)
{
    if (!s) return COLI_E_INVAL;
    if (s->hidden <= 0 || s->hidden % 128 != 0 || s->hidden > 16384) return COLI_E_INVAL;
    if (s->ffn <= 0 || s->ffn % 32 != 0 || s->ffn > 16384) return COLI_E_INVAL;
    if (s->n_experts < 1 || s->n_experts > 256) return COLI_E_INVAL;
    if (s->top_k < 1 || s->top_k > 16 || s->top_k > s->n_experts) return COLI_E_INVAL;
    if (s->max_tok < 1 || s->max_tok > 65536) return COLI_E_INVAL;
    if (!(s->routed_scale > 0.0f) || s->routed_scale > 3.0e38f) return COLI_E_INVAL;
    return COLI_OK;
}

}  // namespace coli

using namespace coli;

extern "C" {

const char *coli_moe_strerror(int code)
{
    switch (code) {
    case COLI_OK: return "ok";
    case COLI_E_INVAL: return "invalid argument";
    case COLI_E_NOSHAPE: return "layer shape not configured";
    case COLI_E_NOMEM: return "workspace allocation failed";
    case COLI_E_CUDA: return "CUDA call or launch failed";
    case COLI_E_TIMEOUT: return "a bounded device-side wait gave up";
    case COLI_E_UNIMPL: return "not implemented";
    case COLI_E_DEVICE: return "device status reports an out-of-range expert index";
    default: return "unknown status";
    }
}

void coli_moe_release(void)
{
    if (g.ws.base || g_tier.pool_w) cudaDeviceSynchronize();
    tier_free();
    free_workspace();
    g.configured = false;
}

void coli_moe_tier_release(void)
{
    if (g_tier.pool_w) cudaDeviceSynchronize();
    tier_free();
}

int coli_moe_tier_configure(int n_slots)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    if (n_slots < 1 || n_slots > g.s.n_experts) return COLI_E_INVAL;
    coli_moe_tier_release();
    const coli_moe_shape &s = g.s;
    Tier t;
    t.n_slots = n_slots;
    t.E = s.n_experts;
    t.wbits = g.wbits;
    t.stride = (size_t)3 * s.ffn * s.hidden * g.wbits / 8;
    t.rs_len = (size_t)2 * s.ffn + s.hidden;
    const size_t n_idx = (size_t)s.max_tok * s.top_k;
    bool ok = cudaMalloc(&t.pool_w, t.stride * n_slots) == cudaSuccess &&
              cudaMalloc(&t.pool_rs, t.rs_len * sizeof(float) * n_slots) == cudaSuccess &&
              cudaMalloc(&t.slot_dev, sizeof(int32_t) * t.E) == cudaSuccess &&
              cudaMallocHost(&t.slot_host, sizeof(int32_t) * t.E) == cudaSuccess &&
              cudaMallocHost(&t.idx_host, sizeof(int32_t) * n_idx) == cudaSuccess;
    if (!ok) {
        (void)cudaGetLastError();
        g_tier = t;
        tier_free();
        return COLI_E_NOMEM;
    }
    if (cudaMemset(t.slot_dev, 0, sizeof(int32_t) * t.E) != cudaSuccess) {
        g_tier = t;
        tier_free();
        return cuda_fail(cudaErrorUnknown);
    }
    t.slot_of.assign(t.E, -1);
    t.expert_in.assign(n_slots, -1);
    t.stamp.assign(n_slots, -1);
    g_tier = std::move(t);
    return COLI_OK;
}

int coli_moe_tier_stats(long long *hits, long long *misses, long long *bytes_h2d, int *resident)
{
    if (!g_tier.pool_w) return COLI_E_NOSHAPE;
    if (hits) *hits = g_tier.hits;
    if (misses) *misses = g_tier.misses;
    if (bytes_h2d) *bytes_h2d = g_tier.bytes;
    if (resident) {
        int n = 0;
        for (int e : g_tier.expert_in) n += e >= 0;
        *resident = n;
    }
    return COLI_OK;
}

int coli_moe_configure(const coli_moe_shape *s)
{
    int st = check_shape(s);
    if (st != COLI_OK) return st;
    coli_moe_release();
    int dev = 0;
    CUDA_OK(cudaGetDevice(&dev));
    int sms = 0;
    CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));

    const size_t T = (size_t)s->max_tok, H = (size_t)s->hidden, F = (size_t)s->ffn;
    const size_t E = (size_t)s->n_experts, k = (size_t)s->top_k;
    const size_t P = T * k, R = P + T;
    const size_t tiles = (size_t)max_gemv_tiles((int)T, (int)k, (int)E);
    const size_t items = (size_t)max_gemm_items((int)T, (int)k, (int)E);
    const size_t Ra = R > 128 ? R : 128;
    // carve one allocation; every piece 256-byte aligned
    struct Piece { void **dst; size_t bytes; };
    Workspace w;
    Piece pieces[] = {
        {(void **)&w.qx, T * H},
        {(void **)&w.dx, T * (H / 32) * 4},
        {(void **)&w.logits, T * E * 4},
        {(void **)&w.sig, T * E * 4},
        {(void **)&w.key, T * E * 4},
        {(void **)&w.idx, P * 4},
        {(void **)&w.wts, P * 4},
        {(void **)&w.counts, E * 4},
        {(void **)&w.offsets, (E + 1) * 4},
        {(void **)&w.perm, P * 4},
        {(void **)&w.inv, P * 4},
        {(void **)&w.pos_token, R * 4},
        {(void **)&w.tile_expert, tiles * 4},
        {(void **)&w.tile_pos0, tiles * 4},
        {(void **)&w.tile_m, tiles * 4},
        {(void **)&w.n_tiles, 4},
        {(void **)&w.sync, (tiles + H / 64 + 2) * 4},
        {(void **)&w.route_counter, 4},
        {(void **)&w.qh, R * F},
        {(void **)&w.dh, R * (F / 32) * 4},
        {(void **)&w.y, R * H * 4},
        {(void **)&w.x_io, T * H * 4},
        {(void **)&w.out_io, T * H * 4},
        {(void **)&w.xn, T * H * 4},
        {(void **)&w.status, 4},
        {(void **)&w.xg, Ra * H * 2},
        {(void **)&w.qhb, Ra * F * 2},
        {(void **)&w.item_expert, items * 4},
        {(void **)&w.item_pos0, items * 4},
        {(void **)&w.item_m, items * 4},
        {(void **)&w.n_items, 4},
    };
    size_t total = WS_GUARD;
    for (auto &p : pieces) total += align_up(p.bytes, 256) + WS_GUARD;
    void *base = nullptr;
    if (g_inj.alloc_fail > 0) {
        --g_inj.alloc_fail;        // injected: behave as a failed cudaMalloc
        return COLI_E_NOMEM;
    }
    if (cudaMalloc(&base, total) != cudaSuccess) {
        (void)cudaGetLastError();
        return COLI_E_NOMEM;
    }
    size_t off = WS_GUARD;
    w.guards.emplace_back(0, WS_GUARD);
    for (auto &p : pieces) {
        *p.dst = (char *)base + off;
        const size_t end = off + align_up(p.bytes, 256) + WS_GUARD;
        w.guards.emplace_back(off + p.bytes, end - (off + p.bytes));
        off = end;
    }
    w.base = base;
    w.bytes = total;
    bool filled = cudaMemset(base, 0, total) == cudaSuccess;
    for (auto &gd : w.guards)
        filled = filled && cudaMemset((char *)base + gd.first, WS_GUARD_BYTE, gd.second) == cudaSuccess;
    if (!filled) {
        cudaFree(base);
        return cuda_fail(cudaErrorUnknown);
    }
    CUDA_OK(cudaDeviceSynchronize());
    w.n_sync = (int)(tiles + H / 64 + 2);
    w.rows_alloc = (int)Ra;
    if (gemm_shape_ok((int)F) && (!encode_act(&g.act_x, w.xg, H, Ra) || !encode_act(&g.act_h, w.qhb, F, Ra))) {
        cudaFree(base);
        return COLI_E_CUDA;
    }
    g.gemm_valid = false;
    g.ws = w;
    g.max_tiles = (int)tiles;
    g.maps_valid = false;
    g.s = *s;
    g.device = dev;
    g.num_sms = sms;
    g.configured = true;
    return COLI_OK;
}

int coli_moe_dbg_inject(int what, long long arg)
{
    switch (what) {
    case COLI_INJECT_NONE:
        g_inj = Inject{};
        return COLI_OK;
    case COLI_INJECT_ALLOC_FAIL:
        if (arg < 0 || arg > 1000000) return COLI_E_INVAL;
        g_inj.alloc_fail = (int)arg;
        return COLI_OK;
    case COLI_INJECT_LAUNCH_FAIL:
        if (arg < 0 || arg > 1000000) return COLI_E_INVAL;
        g_inj.launch_fail_at = (int)arg;
        return COLI_OK;
    case COLI_INJECT_WAIT_TIMEOUT:
        if (arg < 0 || arg > 1000000) return COLI_E_INVAL;
        g_inj.wait_us = arg;
        return COLI_OK;
    case COLI_INJECT_GUARD:
        // host-side: one byte of guard region `arg` changes, as a stray
        // device write past a piece's end would change it
        if (!g.configured) return COLI_E_NOSHAPE;
        if (arg < 0 || arg >= (long long)g.ws.guards.size()) return COLI_E_INVAL;
        CUDA_OK(cudaDeviceSynchronize());
        CUDA_OK(cudaMemset((char *)g.ws.base + g.ws.guards[(size_t)arg].first, 0, 1));
        return COLI_OK;
    default:
        return COLI_E_INVAL;
    }
}

int coli_moe_dbg_check_guards(int *n_guards)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    const auto &gs = g.ws.guards;
    if (n_guards) *n_guards = (int)gs.size();
    CUDA_OK(cudaDeviceSynchronize());
    int bad = 0;
    std::vector<unsigned char> h;
    for (auto &gd : gs) {
        h.resize(gd.second);
        CUDA_OK(cudaMemcpy(h.data(), (char *)g.ws.base + gd.first, gd.second, cudaMemcpyDeviceToHost));
        bool ok = true;
        for (unsigned char c : h) ok = ok && (c == WS_GUARD_BYTE);
        if (!ok) {
            ++bad;
            CUDA_OK(cudaMemset((char *)g.ws.base + gd.first, WS_GUARD_BYTE, gd.second));   // re-arm
        }
    }
    CUDA_OK(cudaDeviceSynchronize());
    return bad;
}

int coli_moe_set_path(int path, int gemm_min_tokens)
{
    if (path < COLI_PATH_AUTO || path > COLI_PATH_GEMM) return COLI_E_INVAL;
    g.path = path;
    g.gemm_min_tokens = gemm_min_tokens;
    return COLI_OK;
}

long long coli_moe_launch_count(void)
{
    long long n = g_launches;
    g_launches = 0;
    return n;
}

int coli_moe_trace_enable(int events_per_block)
{
    if (g.trace) {
        cudaFree(g.trace);
        g.trace = nullptr;
        g.trace_cap = 0;
    }
    if (events_per_block <= 0) return COLI_OK;
    if (events_per_block > 4096) return COLI_E_INVAL;
    int dev = 0, sms = 0;
    CUDA_OK(cudaGetDevice(&dev));
    CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    g.trace_blocks = sms * 32;   // more than any expert-kernel grid
    const size_t bytes = (size_t)g.trace_blocks * events_per_block * 2 * sizeof(unsigned long long);
    if (cudaMalloc(&g.trace, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        g.trace = nullptr;
        return COLI_E_NOMEM;
    }
    CUDA_OK(cudaMemset(g.trace, 0, bytes));
    g.trace_cap = events_per_block;
    return COLI_OK;
}

int coli_moe_trace_read(unsigned long long *host, long long capacity, int *blocks, int *events_per_block)
{
    if (!g.trace) return COLI_E_INVAL;
    const size_t n = (size_t)g.trace_blocks * g.trace_cap * 2;
    if (!host || capacity < (long long)n || !blocks || !events_per_block) return COLI_E_INVAL;
    CUDA_OK(cudaDeviceSynchronize());
    CUDA_OK(cudaMemcpy(host, g.trace, n * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemset(g.trace, 0, n * sizeof(unsigned long long)));
    *blocks = g.trace_blocks;
    *events_per_block = g.trace_cap;
    return COLI_OK;
}

int coli_moe_timing_enable(int on)
{
    g.timing = on != 0;
    return COLI_OK;
}

int coli_moe_timing_read(double *ms_total, int *n_timed)
{
    if (!ms_total || !n_timed) return COLI_E_INVAL;
    double sum = 0.0;
    for (int i = 0; i < g.ev_used; ++i) {
        CUDA_OK(cudaEventSynchronize(g.ev_pool[2 * i + 1]));
        float ms = 0.0f;
        CUDA_OK(cudaEventElapsedTime(&ms, g.ev_pool[2 * i], g.ev_pool[2 * i + 1]));
        sum += ms;
    }
    *ms_total = sum;
    *n_timed = g.ev_used;
    g.ev_used = 0;
    return COLI_OK;
}

static int timing_events(cudaEvent_t *start, cudaEvent_t *stop)
{
    if (g.ev_used * 2 + 2 > (int)g.ev_pool.size()) {
        if (g.ev_pool.size() >= 2 * 65536) return COLI_E_NOMEM;
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t e;
            CUDA_OK(cudaEventCreate(&e));
            g.ev_pool.push_back(e);
        }
    }
    *start = g.ev_pool[2 * g.ev_used];
    *stop = g.ev_pool[2 * g.ev_used + 1];
    ++g.ev_used;
    return COLI_OK;
}

int coli_moe_get_device_status(void *stream)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    cudaStream_t st = (cudaStream_t)stream;
    CUDA_OK(cudaStreamSynchronize(st));
    int v = 0;
    CUDA_OK(cudaMemcpy(&v, g.ws.status, 4, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemset(g.ws.status, 0, 4));
    if (v & ST_TIMEOUT) return COLI_E_TIMEOUT;
    if (v & (ST_BAD_INDEX | ST_BAD_SHAPE)) return COLI_E_DEVICE;
    return COLI_OK;
}

int coli_moe_pack_int4(const float *w, int rows, int K, uint8_t *packed, float *scale, void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return COLI_E_INVAL;
    if (rows == 0) return COLI_OK;
    if (!w || !packed || !scale || ((uintptr_t)w & 7u)) return COLI_E_INVAL;
    LAUNCH_OK(launch_pack_int4(w, rows, K, packed, scale, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_pack_int8(const float *w, int rows, int K, int8_t *q, float *scale, void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return COLI_E_INVAL;
    if (rows == 0) return COLI_OK;
    if (!w || !q || !scale) return COLI_E_INVAL;
    LAUNCH_OK(launch_pack_int8(w, rows, K, q, scale, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_set_weight_bits(int bits)
{
    if (bits != 4 && bits != 8) return COLI_E_INVAL;
    if (bits != g.wbits) {
        g.wbits = bits;
        g.maps_valid = false;
        g.gemm_valid = false;
    }
    return COLI_OK;
}

int coli_moe_dbg_block_dots_w8(const int8_t *w8, int rows, int K, const int8_t *q, int32_t *I_out,
                               void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return COLI_E_INVAL;
    if (rows == 0) return COLI_OK;
    if (!w8 || !q || !I_out || !aligned16(w8) || !aligned16(q)) return COLI_E_INVAL;
    LAUNCH_OK(launch_block_dots_w8(w8, rows, K, q, I_out, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_dbg_quantize(const float *x, int n, int8_t *q, float *d, void *stream)
{
    if (n < 0 || n % 32 != 0) return COLI_E_INVAL;
    if (n == 0) return COLI_OK;
    if (!x || !q || !d) return COLI_E_INVAL;
    LAUNCH_OK(launch_q8_0(x, n, q, d, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_dbg_block_dots(const uint8_t *w4, int rows, int K, const int8_t *q, int32_t *I_out,
                            void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return COLI_E_INVAL;
    if (rows == 0) return COLI_OK;
    if (!w4 || !q || !I_out || !aligned16(w4) || !aligned16(q)) return COLI_E_INVAL;
    LAUNCH_OK(launch_block_dots(w4, rows, K, q, I_out, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_dbg_route(const float *x, int n_tok, const float *router_w, const float *router_bias,
                       int32_t *idx, float *w, float *logits, void *stream)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    const coli_moe_shape &s = g.s;
    if (n_tok < 0 || n_tok > s.max_tok) return COLI_E_INVAL;
    if (n_tok == 0) return COLI_OK;
    if (!x || !router_w || !router_bias || !idx || !w) return COLI_E_INVAL;
    if (!aligned16(x) || !aligned16(router_w)) return COLI_E_INVAL;
    cudaStream_t st = (cudaStream_t)stream;
    float *lg = logits ? logits : g.ws.logits;
    LAUNCH_OK(launch_router_logits(x, n_tok, s.hidden, router_w, s.n_experts, lg, st));
    LAUNCH_OK(launch_topk(lg, n_tok, s.n_experts, s.top_k, router_bias, s.routed_scale, idx, w, st));
    return COLI_OK;
}

int coli_moe_dbg_dispatch(const int32_t *idx, int n_tok, int32_t *counts, int32_t *offsets,
                          int32_t *perm, int32_t *inv, void *stream)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    const coli_moe_shape &s = g.s;
    if (n_tok < 0 || n_tok > s.max_tok) return COLI_E_INVAL;
    if (n_tok == 0) return COLI_OK;
    if (!idx || !counts || !offsets || !perm || !inv) return COLI_E_INVAL;
    Workspace &w = g.ws;
    LAUNCH_OK(launch_dispatch(idx, n_tok, s.top_k, s.n_experts, counts, offsets, perm, inv,
                              w.pos_token, w.tile_expert, w.tile_pos0, w.tile_m, w.n_tiles, w.sync,
                              w.n_sync, w.status, (cudaStream_t)stream));
    return COLI_OK;
}

static int check_forward_args(const float *x, int n_tok, const float *router_w,
                              const float *router_bias, const uint8_t *expert_w4,
                              const float *expert_rowscale, const uint8_t *shared_w4,
                              const float *shared_rowscale, const float *out)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    if (n_tok < 0 || n_tok > g.s.max_tok) return COLI_E_INVAL;
    if (n_tok == 0) return COLI_OK;
    if (!x || !router_w || !router_bias || !expert_w4 || !expert_rowscale || !shared_w4 ||
        !shared_rowscale || !out)
        return COLI_E_INVAL;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(expert_w4) || !aligned16(shared_w4) ||
        !aligned16(out))
        return COLI_E_INVAL;
    if (x == out) return COLI_E_INVAL;
    return COLI_OK;
}

// Argument block of the expert kernel for the configured shape.
static ExpertArgs expert_args(int T, const float *expert_rowscale, const float *shared_rowscale)
{
    const coli_moe_shape &s = g.s;
    Workspace &w = g.ws;
    ExpertArgs a{};
    a.H = s.hidden; a.F = s.ffn; a.E = s.n_experts; a.k = s.top_k;
    a.n_tok = T; a.P = T * s.top_k;
    a.KC = stage_kc(s.hidden, s.ffn, g.wbits);
    a.wbits = g.wbits;
    a.gate_up_only = 0;
    a.expert_rs = expert_rowscale; a.shared_rs = shared_rowscale;
    a.shared_w4 = nullptr;
    a.qx = w.qx; a.dx = w.dx; a.pos_token = w.pos_token;
    a.tile_expert = w.tile_expert; a.tile_pos0 = w.tile_pos0; a.tile_m = w.tile_m;
    a.n_tiles = w.n_tiles;
    a.inv = w.inv; a.wts = w.wts;
    a.qh = w.qh; a.dh = w.dh; a.h_dbg = nullptr; a.y = w.y; a.out = nullptr; a.res = nullptr;
    a.g_done = w.sync;
    a.w_done = w.sync + g.max_tiles;
    a.work_counter = w.sync + g.max_tiles + s.hidden / 64;
    a.blocks_done = a.work_counter + 1;
    a.sync_base = w.sync;
    a.n_sync = w.n_sync;
    a.status = w.status;
    a.trace = g.trace;
    a.trace_cap = g.trace_cap;
    a.wait_ns = 2000000000ull;     // 2 s
    a.gdone_extra = 0;
    a.next_rw = a.next_sw = nullptr;
    a.next_rw_bytes = a.next_sw_bytes = 0;
    return a;
}

// The forward, in three phases: the plan (expert path and weight maps), the
// routing launches, and the expert launches.  `n_w` is the extent of the
// routed-weight arrays (E, or the slots of the host-memory tier, whose
// `slot_of` table maps each routed expert to its slot).
struct FwdPlan {
    bool use_gemm = false;
    ExpertMaps maps{};
};

static int plan_forward(int T, const uint8_t *expert_w4, int n_w, const uint8_t *shared_w4, FwdPlan *p)
{
    const coli_moe_shape &s = g.s;
    const int E = s.n_experts, k = s.top_k;
    const bool big = g.gemm_min_tokens > 0 ? T >= g.gemm_min_tokens
                                           : (long)T * k >= (long)COLI_GEMM_MIN_PAIRS_PER_EXPERT * E;
    const bool gemm_ok = gemm_shape_ok(s.ffn);
    if (g.path == COLI_PATH_GEMM && !gemm_ok) return COLI_E_UNIMPL;
    p->use_gemm = g.path == COLI_PATH_GEMM || (g.path == COLI_PATH_AUTO && big && gemm_ok);
    if (p->use_gemm) {
        if (!gemm_weight_maps(expert_w4, n_w, shared_w4)) return COLI_E_CUDA;
    } else if (!expert_maps(expert_w4, n_w, shared_w4, &p->maps)) {
        return COLI_E_CUDA;
    }
    return COLI_OK;
}

static int route_phase(const float *x, int T, const float *router_w, const float *router_bias, cudaStream_t st)
{
    const coli_moe_shape &s = g.s;
    Workspace &w = g.ws;
    const int H = s.hidden, E = s.n_experts, k = s.top_k;
    if (T <= ROUTE_SMALL_MAX_T) {
        RouteArgs r{};
        r.x = x; r.T = T; r.H = H; r.E = E; r.k = k; r.routed_scale = s.routed_scale;
        r.W = router_w; r.bias = router_bias;
        r.qx = w.qx; r.dx = w.dx; r.logits = w.logits; r.idx = w.idx; r.wts = w.wts;
        r.sig = w.sig; r.key = w.key;
        r.counts = w.counts; r.offsets = w.offsets; r.perm = w.perm; r.inv = w.inv;
        r.pos_token = w.pos_token;
        r.tile_expert = w.tile_expert; r.tile_pos0 = w.tile_pos0; r.tile_m = w.tile_m;
        r.n_tiles = w.n_tiles; r.sync = w.sync; r.n_sync = w.n_sync;
        r.route_counter = w.route_counter; r.status = w.status;
        // routing-tail phase stamps go to the last block's slots of the trace log
        r.trace = g.trace ? g.trace + (size_t)(g.trace_blocks - 1) * g.trace_cap * 2 : nullptr;
        LAUNCH_OK(launch_route_small(r, st));
    } else {
        LAUNCH_OK(launch_q8_0(x, (long)T * H, w.qx, w.dx, st));
        LAUNCH_OK(launch_router_logits(x, T, H, router_w, E, w.logits, st));
        LAUNCH_OK(launch_topk(w.logits, T, E, k, router_bias, s.routed_scale, w.idx, w.wts, st));
        LAUNCH_OK(launch_dispatch(w.idx, T, k, E, w.counts, w.offsets, w.perm, w.inv, w.pos_token,
                                  w.tile_expert, w.tile_pos0, w.tile_m, w.n_tiles, w.sync, w.n_sync,
                                  w.status, st));
    }
    return COLI_OK;
}

static int expert_phase(const FwdPlan &p, int T, const float *expert_rowscale, const uint8_t *shared_w4,
                        const float *shared_rowscale, float *out, cudaStream_t st, const float *res,
                        const float *next_rw, const uint8_t *next_sw, const int32_t *slot_of)
{
    const coli_moe_shape &s = g.s;
    Workspace &w = g.ws;
    const int H = s.hidden, E = s.n_experts, k = s.top_k;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (p.use_gemm) {
        const int P = T * k, F = s.ffn;
        LAUNCH_OK(launch_gather_x(w.qx, w.pos_token, w.offsets, E, P, P + T, T, H, w.xg, w.status, st));
        LAUNCH_OK(launch_gemm_items(w.counts, w.offsets, E, T, P, w.item_expert, w.item_pos0, w.item_m,
                                    w.n_items, st));
        GemmArgs ga{};
        ga.H = H; ga.F = F; ga.E = E; ga.T = T;
        ga.n_items = w.n_items; ga.item_expert = w.item_expert; ga.item_pos0 = w.item_pos0;
        ga.item_m = w.item_m; ga.pos_token = w.pos_token; ga.dx = w.dx;
        ga.expert_rs = expert_rowscale; ga.shared_rs = shared_rowscale;
        ga.qh = w.qh; ga.dh = w.dh; ga.qhb = w.qhb; ga.h_dbg = nullptr; ga.y = w.y;
        ga.status = w.status;
        ga.slot_of = slot_of;
        ga.trace = g.trace;            // the stage log covers the gate/up launch
        ga.trace_cap = g.trace_cap;
        if (g.timing) {
            int r = timing_events(&e0, &e1);
            if (r != COLI_OK) return r;
            CUDA_OK(cudaEventRecord(e0, st));
        }
        LAUNCH_OK(launch_gemm(true, g.wbits, g.gemm_gu, ga, g.num_sms, st));
        if (g.timing) CUDA_OK(cudaEventRecord(e1, st));
        ga.trace = nullptr;
        LAUNCH_OK(launch_gemm(false, g.wbits, g.gemm_dn, ga, g.num_sms, st));
        LAUNCH_OK(launch_combine(w.y, w.inv, w.wts, T, k, P, H, res, out, st));
        return COLI_OK;
    }

    ExpertArgs a = expert_args(T, expert_rowscale, shared_rowscale);
    a.out = out;
    a.res = res;
    a.shared_w4 = shared_w4;
    a.slot_of = slot_of;
    if (next_rw) {
        a.next_rw = reinterpret_cast<const unsigned char *>(next_rw);
        a.next_rw_bytes = (size_t)E * H * sizeof(float);
    }
    if (next_sw) {
        a.next_sw = next_sw;
        a.next_sw_bytes = (size_t)3 * s.ffn * H * g.wbits / 8;
    }
    if (g_inj.wait_us > 0) {
        // injected: every down unit waits for one gate/up unit more than its
        // tile has, so each wait runs out after the short bound
        a.wait_ns = (unsigned long long)g_inj.wait_us * 1000ull;
        a.gdone_extra = 1;
        g_inj.wait_us = 0;
    }
    if (g.timing) {
        int r = timing_events(&e0, &e1);
        if (r != COLI_OK) return r;
        CUDA_OK(cudaEventRecord(e0, st));
    }
    LAUNCH_OK(launch_experts(p.maps, a, g.num_sms, st));
    if (g.timing) CUDA_OK(cudaEventRecord(e1, st));
    return COLI_OK;
}

static int forward_impl(const float *x, int n_tok, const float *router_w, const float *router_bias,
                        const uint8_t *expert_w4, const float *expert_rowscale,
                        const uint8_t *shared_w4, const float *shared_rowscale, float *out,
                        cudaStream_t st, const float *res = nullptr, const float *next_rw = nullptr,
                        const uint8_t *next_sw = nullptr)
{
    FwdPlan p;
    int r = plan_forward(n_tok, expert_w4, g.s.n_experts, shared_w4, &p);
    if (r != COLI_OK) return r;
    r = route_phase(x, n_tok, router_w, router_bias, st);
    if (r != COLI_OK) return r;
    return expert_phase(p, n_tok, expert_rowscale, shared_w4, shared_rowscale, out, st, res, next_rw, next_sw,
                        nullptr);
}

int coli_moe_tier_forward(const float *x, int n_tok, const float *router_w, const float *router_bias,
                          const uint8_t *host_expert_w, const float *host_expert_rowscale,
                          const uint8_t *shared_w4, const float *shared_rowscale, float *out, void *stream)
{
    if (!g.configured || !g_tier.pool_w) return COLI_E_NOSHAPE;
    Tier &t = g_tier;
    if (t.wbits != g.wbits || t.E != g.s.n_experts) return COLI_E_INVAL;   // reconfigure the tier
    int st = check_forward_args(x, n_tok, router_w, router_bias, t.pool_w, t.pool_rs, shared_w4,
                                shared_rowscale, out);
    if (st != COLI_OK || n_tok == 0) return st;
    if (!host_expert_w || !host_expert_rowscale) return COLI_E_INVAL;
    cudaStream_t cs = (cudaStream_t)stream;
    const int k = g.s.top_k, E = t.E;
    FwdPlan p;
    st = plan_forward(n_tok, t.pool_w, t.n_slots, shared_w4, &p);
    if (st != COLI_OK) return st;
    st = route_phase(x, n_tok, router_w, router_bias, cs);
    if (st != COLI_OK) return st;
    // the routing's expert choices, on the host
    CUDA_OK(cudaMemcpyAsync(t.idx_host, g.ws.idx, sizeof(int32_t) * n_tok * k, cudaMemcpyDeviceToHost, cs));
    CUDA_OK(cudaStreamSynchronize(cs));
    std::vector<char> need(E, 0);
    int n_need = 0;
    for (int i = 0; i < n_tok * k; ++i) {
        const int e = t.idx_host[i];
        if (e >= 0 && e < E && !need[e]) {   // an index out of range is the kernels' to report
            need[e] = 1;
            ++n_need;
        }
    }
    if (n_need > t.n_slots) return COLI_E_INVAL;      // one forward's union must fit in the slots
    ++t.clock;
    for (int e = 0; e < E; ++e)
        if (need[e] && t.slot_of[e] >= 0) {
            ++t.hits;
            t.stamp[t.slot_of[e]] = t.clock;
        }
    for (int e = 0; e < E; ++e) {
        if (!need[e] || t.slot_of[e] >= 0) continue;
        // least recently used slot not taken by this forward (empty slots first)
        int v = -1;
        for (int q = 0; q < t.n_slots; ++q)
            if (t.stamp[q] < t.clock && (v < 0 || t.stamp[q] < t.stamp[v])) v = q;
        if (v < 0) return COLI_E_INVAL;
        if (t.expert_in[v] >= 0) t.slot_of[t.expert_in[v]] = -1;
        CUDA_OK(cudaMemcpyAsync(t.pool_w + (size_t)v * t.stride, host_expert_w + (size_t)e * t.stride, t.stride,
                                cudaMemcpyHostToDevice, cs));
        CUDA_OK(cudaMemcpyAsync(t.pool_rs + (size_t)v * t.rs_len, host_expert_rowscale + (size_t)e * t.rs_len,
                                t.rs_len * sizeof(float), cudaMemcpyHostToDevice, cs));
        t.slot_of[e] = v;
        t.expert_in[v] = e;
        t.stamp[v] = t.clock;
        ++t.misses;
        t.bytes += (long long)(t.stride + t.rs_len * sizeof(float));
    }
    for (int e = 0; e < E; ++e) t.slot_host[e] = t.slot_of[e] >= 0 ? t.slot_of[e] : 0;
    CUDA_OK(cudaMemcpyAsync(t.slot_dev, t.slot_host, sizeof(int32_t) * E, cudaMemcpyHostToDevice, cs));
    return expert_phase(p, n_tok, t.pool_rs, shared_w4, shared_rowscale, out, cs, nullptr, nullptr, nullptr,
                        t.slot_dev);
}

int coli_moe_layer_forward(const float *x, int n_tok, const float *router_w,
                           const float *router_bias, const uint8_t *expert_w4,
                           const float *expert_rowscale, const uint8_t *shared_w4,
                           const float *shared_rowscale, float *out, void *stream)
{
    int st = check_forward_args(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale,
                                shared_w4, shared_rowscale, out);
    if (st != COLI_OK || n_tok == 0) return st;
    return forward_impl(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                        shared_rowscale, out, (cudaStream_t)stream);
}

int coli_moe_layer_forward_residual(const float *x, int n_tok, const float *router_w,
                                    const float *router_bias, const uint8_t *expert_w4,
                                    const float *expert_rowscale, const uint8_t *shared_w4,
                                    const float *shared_rowscale, float *out, void *stream)
{
    int st = check_forward_args(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale,
                                shared_w4, shared_rowscale, out);
    if (st != COLI_OK || n_tok == 0) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    LAUNCH_OK(launch_rmsnorm(x, n_tok, g.s.hidden, RMSNORM_EPS, g.ws.xn, cs));
    return forward_impl(g.ws.xn, n_tok, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                        shared_rowscale, out, cs, x);
}

int coli_moe_layer_forward_residual_prefetch(const float *x, int n_tok, const float *router_w,
                                             const float *router_bias, const uint8_t *expert_w4,
                                             const float *expert_rowscale, const uint8_t *shared_w4,
                                             const float *shared_rowscale, const float *next_router_w,
                                             const uint8_t *next_shared_w4, float *out, void *stream)
{
    int st = check_forward_args(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale,
                                shared_w4, shared_rowscale, out);
    if (st != COLI_OK || n_tok == 0) return st;
    if ((next_router_w && !aligned16(next_router_w)) || (next_shared_w4 && !aligned16(next_shared_w4)))
        return COLI_E_INVAL;
    cudaStream_t cs = (cudaStream_t)stream;
    LAUNCH_OK(launch_rmsnorm(x, n_tok, g.s.hidden, RMSNORM_EPS, g.ws.xn, cs));
    return forward_impl(g.ws.xn, n_tok, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                        shared_rowscale, out, cs, x, next_router_w, next_shared_w4);
}

int coli_moe_dbg_rmsnorm(const float *x, int n_tok, int hidden, float *xn, void *stream)
{
    if (n_tok < 0 || hidden <= 0 || hidden % 4 != 0) return COLI_E_INVAL;
    if (n_tok == 0) return COLI_OK;
    if (!x || !xn || !aligned16(x) || !aligned16(xn)) return COLI_E_INVAL;
    LAUNCH_OK(launch_rmsnorm(x, n_tok, hidden, RMSNORM_EPS, xn, (cudaStream_t)stream));
    return COLI_OK;
}

int coli_moe_dbg_stream_read(const void *buf, size_t bytes, int chunk, int stages, int blocks_per_sm,
                             unsigned long long *sum, void *stream)
{
    if (!buf || !sum || !aligned16(buf) || bytes % 16 != 0 || ((uintptr_t)sum & 7) != 0) return COLI_E_INVAL;
    if (chunk == 0) chunk = 16384;
    if (stages == 0) stages = 3;
    if (blocks_per_sm == 0) blocks_per_sm = 4;
    // chunks of 1-64 KB in 1 KB steps, 2-16 stages, at most 200 KB of ring per block
    if (chunk < 1024 || chunk > 65536 || chunk % 1024 != 0 || stages < 2 || stages > 16 ||
        (long)chunk * stages > 200L * 1024 || blocks_per_sm < 1 || blocks_per_sm > 32)
        return COLI_E_INVAL;
    cudaStream_t s = (cudaStream_t)stream;
    int dev = 0, sms = 0, smem_sm = 0;
    CUDA_OK(cudaGetDevice(&dev));
    CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CUDA_OK(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
    // every block resident at once (1 KB of each block's shared memory is the system's)
    if ((long)blocks_per_sm * ((long)chunk * stages + 2048) > smem_sm) return COLI_E_INVAL;
    CUDA_OK(cudaMemsetAsync(sum, 0, sizeof(unsigned long long), s));
    if (bytes == 0) return COLI_OK;
    LAUNCH_OK(launch_stream_read(buf, bytes, chunk, stages, blocks_per_sm, sum, nullptr, sms, s));
    return COLI_OK;
}

int coli_moe_layer_forward_hostio(const float *x_host, int n_tok, const float *router_w,
                                  const float *router_bias, const uint8_t *expert_w4,
                                  const float *expert_rowscale, const uint8_t *shared_w4,
                                  const float *shared_rowscale, float *out_host, void *stream)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    if (!x_host || !out_host) return COLI_E_INVAL;
    int st = check_forward_args(g.ws.x_io, n_tok, router_w, router_bias, expert_w4,
                                expert_rowscale, shared_w4, shared_rowscale, g.ws.out_io);
    if (st != COLI_OK || n_tok == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t bytes = (size_t)n_tok * g.s.hidden * sizeof(float);
    // Page-locked, device-mapped output (pinned memory on this platform):
    // the combine writes the result straight into it over the host link,
    // which saves a copy-out launch.  Any other host memory gets the
    // device-side result copied out.
    float *out_mapped = nullptr;
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer && aligned16(pa.devicePointer))
        out_mapped = static_cast<float *>(pa.devicePointer);
    else
        (void)cudaGetLastError();   // an unregistered pointer leaves an error to clear
    CUDA_OK(cudaMemcpyAsync(g.ws.x_io, x_host, bytes, cudaMemcpyHostToDevice, s));
    st = forward_impl(g.ws.x_io, n_tok, router_w, router_bias, expert_w4, expert_rowscale,
                      shared_w4, shared_rowscale, out_mapped ? out_mapped : g.ws.out_io, s);
    if (st != COLI_OK) return st;
    if (!out_mapped) CUDA_OK(cudaMemcpyAsync(out_host, g.ws.out_io, bytes, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    return COLI_OK;
}

int coli_moe_dbg_forward_intermediates(const float *x, int n_tok, const float *router_w,
                                       const float *router_bias, const uint8_t *expert_w4,
                                       const float *expert_rowscale, const uint8_t *shared_w4,
                                       const float *shared_rowscale, float *out, int8_t *qx,
                                       float *dx, int32_t *idx, float *wts, int8_t *qh, float *dh,
                                       float *y, void *stream)
{
    int st = check_forward_args(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale,
                                shared_w4, shared_rowscale, out);
    if (st != COLI_OK || n_tok == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = forward_impl(x, n_tok, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                      shared_rowscale, out, s);
    if (st != COLI_OK) return st;
    const coli_moe_shape &sh = g.s;
    Workspace &w = g.ws;
    const size_t T = (size_t)n_tok, H = sh.hidden, F = sh.ffn, k = sh.top_k;
    if (qx) CUDA_OK(cudaMemcpyAsync(qx, w.qx, T * H, cudaMemcpyDeviceToDevice, s));
    if (dx) CUDA_OK(cudaMemcpyAsync(dx, w.dx, T * (H / 32) * 4, cudaMemcpyDeviceToDevice, s));
    if (idx) CUDA_OK(cudaMemcpyAsync(idx, w.idx, T * k * 4, cudaMemcpyDeviceToDevice, s));
    if (wts) CUDA_OK(cudaMemcpyAsync(wts, w.wts, T * k * 4, cudaMemcpyDeviceToDevice, s));
    if (qh || dh || y)
        LAUNCH_OK(launch_gather_pairs(w.inv, n_tok, sh.top_k, n_tok * sh.top_k, w.qh, w.dh, w.y,
                                      (int)F, (int)H, qh, dh, y, s));
    return COLI_OK;
}

int coli_moe_dbg_expert_hidden(const uint8_t *ew4, const float *ers, const int8_t *qx,
                               const float *dx, int n, float *h, int8_t *qh, float *dh,
                               void *stream)
{
    if (!g.configured) return COLI_E_NOSHAPE;
    const coli_moe_shape &s = g.s;
    if (n < 1 || n > s.max_tok) return COLI_E_INVAL;
    if (!ew4 || !ers || !qx || !dx || !h || !qh || !dh) return COLI_E_INVAL;
    if (!aligned16(ew4) || !aligned16(qx)) return COLI_E_INVAL;
    cudaStream_t st = (cudaStream_t)stream;
    Workspace &w = g.ws;
    ExpertMaps maps;
    if (!expert_maps(ew4, 1, ew4, &maps)) return COLI_E_CUDA;
    LAUNCH_OK(launch_single_expert_tiles(n, w.pos_token, w.tile_expert, w.tile_pos0, w.tile_m,
                                         w.n_tiles, w.sync, w.n_sync, st));
    ExpertArgs a = expert_args(n, ers, ers);
    a.E = 1;   // the one expert is tile expert 0, read through the routed map
    a.k = 1;
    a.P = 0;
    a.qx = qx; a.dx = dx;
    a.qh = qh; a.dh = dh; a.h_dbg = h;
    a.gate_up_only = 1;
    LAUNCH_OK(launch_experts(maps, a, g.num_sms, st));
    g.maps_valid = false;   // the maps above describe a single expert
    return COLI_OK;
}

}  // extern "C"
