// coli_internal.h -- host-side declarations shared by the library's
// translation units (launchers and the argument blocks of the kernels).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace coli {

// Tensor maps of the expert weights (3-D: bytes of a row, rows, expert).
struct ExpertMaps {
    CUtensorMap gu;    // routed gate/up rows [E][2F][H/2], box KC x 32 x 1
    CUtensorMap dn;    // routed down rows    [E][H][F/2],  box KC x 64 x 1
    CUtensorMap sgu;   // shared expert gate/up
    CUtensorMap sdn;   // shared expert down
};

// Per-forward view of the workspace and the weights, passed by value to the
// expert kernel.
struct ExpertArgs {
    int H, F, E, k;
    int n_tok;                      // T
    int P;                          // T * k (routed pairs); shared rows follow at P + t
    int KC;                         // bytes of a weight row per TMA box (128, 64, 32 or 16)
    int wbits;                      // weight container: 4 (packed int4) or 8 (int8 codes)
    int nstage;                     // ring depth (set by the launcher)
    int gate_up_only;               // 1: stop after h (stage tests)
    const float *expert_rs;         // [E][2F+H]
    const float *shared_rs;         // [2F+H]
    const uint8_t *shared_w4;       // [3FH/2] packed shared expert (prefetched into L2 during routing)
    const int8_t *qx;               // [T][H]
    const float *dx;                // [T][H/32]
    const int32_t *pos_token;       // [P+T] token of each dispatch position
    const int32_t *tile_expert;     // [n_tiles] expert (E = shared)
    const int32_t *tile_pos0;       // [n_tiles] first dispatch position
    const int32_t *tile_m;          // [n_tiles] tokens in the tile (1..GEMV_MT)
    const int32_t *n_tiles;         // device scalar
    const int32_t *inv;             // [P] position of each pair
    const float *wts;               // [P] routed weights
    int8_t *qh;                     // [P+T][F] requantised hidden, by position
    float *dh;                      // [P+T][F/32]
    float *h_dbg;                   // optional [P+T][F] hidden before requantisation
    float *y;                       // [P+T][H] expert outputs, by position
    float *out;                     // [T][H]
    const float *res;               // optional [T][H] residual: out = res + layer output
    int *g_done;                    // [n_tiles] finished gate/up units per tile
    int *w_done;                    // [H/64] finished down units per row chunk
    int *work_counter;              // next unit to claim
    int *blocks_done;               // blocks that finished (the last one resets)
    int *sync_base;                 // all of the above counters, n_sync ints
    int n_sync;
    int *status;
    unsigned long long *trace;      // optional per-block event log (null: off)
    int trace_cap;                  // events per block
    unsigned long long wait_ns;     // bound of a down unit's wait for its tile's gate/up units
    int gdone_extra;                // test injection: added to the gate/up count that wait needs (0)
    // layer-ahead L2 prefetch (stacked decode): the next layer's router
    // weights and shared expert, pulled into L2 by blocks that ran out of units
    const unsigned char *next_rw;   // null: none
    size_t next_rw_bytes;
    const unsigned char *next_sw;   // null: none
    size_t next_sw_bytes;
    const int32_t *slot_of;         // optional [E]: routed expert e lives at index slot_of[e] of
                                    // expert_w4 / expert_rs (host-memory tier); null: at index e
};

// Tensor maps of one grouped-GEMM launch: the bf16 activation codes by
// dispatch position (2-D, box 64 x 128, 128-byte swizzle) and the packed
// weight rows of the routed experts and of the shared expert (3-D, box of 64
// weights' bytes x 128 or 256 rows x 1, no swizzle).
struct GemmMaps {
    CUtensorMap act;
    CUtensorMap w;
    CUtensorMap sw;
};

// Argument block of the grouped-GEMM kernels (gate/up and down).
struct GemmArgs {
    int H, F, E, T;
    const int32_t *n_items;          // device scalar
    const int32_t *item_expert;      // [n_items] expert (E = shared)
    const int32_t *item_pos0;        // [n_items] first dispatch position
    const int32_t *item_m;           // [n_items] positions in the item (1..128)
    const int32_t *pos_token;        // [P+T]
    const float *dx;                 // [T][H/32] activation block scales
    const float *expert_rs;          // [E][2F+H]
    const float *shared_rs;          // [2F+H]
    int8_t *qh;                      // [P+T][F] requantised hidden, by position
    float *dh;                       // [P+T][F/32]
    uint16_t *qhb;                   // [P+T][F] the same codes as bf16 (down-GEMM operand)
    float *h_dbg;                    // optional [P+T][F]
    float *y;                        // [P+T][H]
    int *status;
    const int32_t *slot_of;          // optional [E]: index of routed expert e in the weight arrays
    unsigned long long *trace;       // optional per-block stage log (null: off)
    int trace_cap;                   // events per block (four roles, a quarter each)
};

// Small-batch routing in one launch: Q8_0 of x, router logits, top-k, dispatch,
// tile list, and zeroing of the expert kernel's counters.
struct RouteArgs {
    const float *x;
    int T, H, E, k;
    float routed_scale;
    const float *W;
    const float *bias;
    int8_t *qx;
    float *dx;
    float *logits;
    float *sig, *key;               // [T][E] sigma and selection key (sigma + bias)
    int32_t *idx;
    float *wts;
    int32_t *counts, *offsets, *perm, *inv, *pos_token;
    int32_t *tile_expert, *tile_pos0, *tile_m, *n_tiles;
    int *sync;                      // expert-kernel counters to zero
    int n_sync;
    int *route_counter;             // blocks finished (reset by the last block)
    int *status;
    unsigned long long *trace;      // optional phase log of the routing tail (null: off)
};
constexpr int ROUTE_SMALL_MAX_T = 8;

void count_launch();

int launch_q8_0(const float *x, long n, int8_t *q, float *d, cudaStream_t st);
// Pre-norm of a stacked layer (xn = x / sqrt(mean(x^2) + eps) per token).
constexpr float RMSNORM_EPS = 1e-6f;
int launch_rmsnorm(const float *x, int T, int H, float eps, float *xn, cudaStream_t st);
int launch_pack_int4(const float *w, int rows, int K, uint8_t *packed, float *scale, cudaStream_t st);
int launch_pack_int8(const float *w, int rows, int K, int8_t *q, float *scale, cudaStream_t st);
int launch_block_dots(const uint8_t *w4, int rows, int K, const int8_t *q, int32_t *I, cudaStream_t st);
int launch_block_dots_w8(const int8_t *w8, int rows, int K, const int8_t *q, int32_t *I, cudaStream_t st);
int launch_stream_read(const void *buf, size_t bytes, int chunk, int stages, int blocks_per_sm,
                       unsigned long long *sum, int *status, int num_sms, cudaStream_t st);

int launch_router_logits(const float *x, int T, int H, const float *W, int E, float *logits,
                         cudaStream_t st);
int launch_topk(const float *logits, int T, int E, int k, const float *bias, float routed_scale,
                int32_t *idx, float *w, cudaStream_t st);
// Stable counting sort of the T*k pairs by expert, the GEMV tile list (shared
// expert first, then routed experts in ascending id), and zeroing of `sync`.
int launch_dispatch(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv, int32_t *pos_token, int32_t *tile_expert,
                    int32_t *tile_pos0, int32_t *tile_m, int32_t *n_tiles, int *sync, int n_sync,
                    int *status, cudaStream_t st);
int launch_route_small(const RouteArgs &r, cudaStream_t st);
// Tile list for one expert over n consecutive positions (stage tests).
int launch_single_expert_tiles(int n, int32_t *pos_token, int32_t *tile_expert, int32_t *tile_pos0,
                               int32_t *tile_m, int32_t *n_tiles, int *sync, int n_sync,
                               cudaStream_t st);

int max_gemv_tiles(int T, int k, int E);
size_t experts_smem_bytes(int H, int F);
int launch_experts(const ExpertMaps &maps, const ExpertArgs &a, int num_sms, cudaStream_t st);
int launch_gather_pairs(const int32_t *inv, int T, int k, int P, const int8_t *qh, const float *dh,
                        const float *y, int F, int H, int8_t *qh_out, float *dh_out, float *y_out,
                        cudaStream_t st);

// Grouped tensor-core path.
int max_gemm_items(int T, int k, int E);
int gemm_tile_rows();
size_t gemm_smem_bytes();
int launch_gather_x(const int8_t *qx, const int32_t *pos_token, const int32_t *offsets, int E, int P, int R,
                    int T, int H, uint16_t *xg, int *status, cudaStream_t st);
int launch_gemm_items(const int32_t *counts, const int32_t *offsets, int E, int T, int P, int32_t *item_expert,
                      int32_t *item_pos0, int32_t *item_m, int32_t *n_items, cudaStream_t st);
int launch_gemm(bool gateup, int wbits, const GemmMaps &maps, const GemmArgs &g, int num_sms, cudaStream_t st);
int launch_combine(const float *y, const int32_t *inv, const float *wts, int T, int k, int P, int H,
                   const float *res, float *out, cudaStream_t st);

}  // namespace coli
