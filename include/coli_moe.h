/*
 * coli_moe.h -- C ABI of the GB300 (sm_103a) quantized MoE feed-forward layer.
 *
 * The layer (a GLM-5.2-class MoE FFN as the colibri pages describe it):
 *   - a DeepSeek-V3-style F32 sigmoid router over E routed experts picks top-k
 *     experts per token ("Open-source engine that ran 744B GLM-5.2 on a
 *     25GB-RAM laptop" (jeff.news), section "Attention and kernels"; router in
 *     F32: "GLM-5.2-colibri-int4" model card, section "Good to know");
 *   - one shared expert runs on every token (same section);
 *   - each expert is a SwiGLU FFN whose weights are packed int4 nibbles, two
 *     per byte, with a per-row F32 scale (model card, "Technical features");
 *   - activations are quantized Q8_0-style (blocks of 32, int8 codes, one F32
 *     scale, lrintf rounding) and every matmul is an integer dot product
 *     accumulated in int32 per block, then scaled in float ("colibri: a pure-C
 *     inference engine ..." (discuss.pytorch.kr), section "Key features").
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers owned by the caller (except the
 *     *_host arguments of coli_moe_layer_forward_hostio).  The library never
 *     frees or retains them beyond the call's GPU work.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously; no entry point synchronises the host
 *     unless it says so.
 *   - Row-major, contiguous layouts.  Int4 matrices [N][K] are N*K/2 bytes:
 *     byte j of a row holds element 2j in its low nibble and element 2j+1 in its
 *     high nibble, each stored as code + 8 (codes -7..7; a nibble of 0 decodes
 *     to -8 and is accepted).
 *   - One expert is gate [F][H], up [F][H], down [H][F] back to back
 *     (3*F*H/2 bytes); its row scales are [gate F | up F | down H] F32.
 *     expert_w4 is [E][3*F*H/2], expert_rowscale is [E][2F+H]; the shared
 *     expert has the same layout without the E dimension.
 *   - Return value: COLI_OK or a negative coli_status.  Argument errors are
 *     reported before anything is launched.  A launch failure returns
 *     COLI_E_CUDA after clearing the CUDA error state.  Device-side problems
 *     (an expert index out of range, a bounded wait that gave up) set a device
 *     status word that coli_moe_get_device_status() reads.
 *   - Not thread-safe: one host thread drives the library at a time.
 */
#ifndef COLI_MOE_H
#define COLI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    COLI_OK = 0,
    COLI_E_INVAL = -1,     /* bad argument: NULL, misaligned, out of range   */
    COLI_E_NOSHAPE = -2,   /* coli_moe_configure() has not succeeded yet      */
    COLI_E_NOMEM = -3,     /* workspace allocation failed                     */
    COLI_E_CUDA = -4,      /* a CUDA call or launch failed                    */
    COLI_E_TIMEOUT = -5,   /* a bounded device-side wait gave up              */
    COLI_E_UNIMPL = -6,    /* requested path or shape not implemented         */
    COLI_E_DEVICE = -7     /* device status word reports a bad index          */
} coli_status;

/* Layer shape.  Limits: hidden % 128 == 0, ffn % 32 == 0, 1 <= top_k <= 16,
 * top_k <= n_experts <= 256, 1 <= max_tok <= 65536, routed_scale finite > 0.
 * The grouped tensor-core path needs ffn % 128 == 0: with another ffn, AUTO
 * always takes the streaming path and COLI_PATH_GEMM forwards return
 * COLI_E_UNIMPL. */
typedef struct {
    int hidden;          /* H: model width                                     */
    int ffn;             /* F: expert FFN width                                */
    int n_experts;       /* E: routed experts                                  */
    int top_k;           /* k: experts per token                               */
    float routed_scale;  /* multiplier of the renormalised routed weights      */
    int max_tok;         /* largest n_tok any later call will pass             */
} coli_moe_shape;

/* Execution path of the expert matmuls.  Both give bit-identical results. */
typedef enum {
    COLI_PATH_AUTO = 0,  /* per forward: GEMM when n_tok >= the threshold       */
    COLI_PATH_GEMV = 1,  /* streaming int4 x int8 dp4a kernels (decode batches) */
    COLI_PATH_GEMM = 2   /* tcgen05 grouped GEMM over the batch union (prefill) */
} coli_path;

/* Validate `s`, remember it and allocate the library-owned workspace for up to
 * s->max_tok tokens on the current CUDA device (replacing an earlier one).
 * Returns COLI_E_INVAL for a shape outside the limits, COLI_E_NOMEM if the
 * workspace cannot be allocated.  Synchronises the device. */
int coli_moe_configure(const coli_moe_shape *s);

/* One MoE layer forward on n_tok tokens (0 <= n_tok <= max_tok; 0 is a no-op).
 *   x               [n_tok][H] F32 input activations (16-byte aligned)
 *   router_w        [E][H] F32, router_bias [E] F32
 *   expert_w4       [E][3FH/2] packed int4 (16-byte aligned)
 *   expert_rowscale [E][2F+H] F32
 *   shared_w4       [3FH/2] packed int4 (16-byte aligned)
 *   shared_rowscale [2F+H] F32
 *   out             [n_tok][H] F32 output: shared expert + sum over the top-k of
 *                   w_r * expert_r(x), w_r = sigma_r / sum(sigma_sel) * routed_scale.
 * Steps, all on `stream`: Q8_0-quantise x; route (logits in a fixed F32
 * order, sigmoid, +bias for selection, top-k, renormalise); build the stable
 * token->expert permutation; gate/up with SiLU*up and Q8_0 requantisation;
 * down; gate-weighted combine.  Asynchronous; `out` may not alias `x`. */
int coli_moe_layer_forward(const float *x, int n_tok,
                           const float *router_w, const float *router_bias,
                           const uint8_t *expert_w4, const float *expert_rowscale,
                           const uint8_t *shared_w4, const float *shared_rowscale,
                           float *out, void *stream);

/* The forward of one layer of a stacked decoder (the multi-layer sweep of
 * the benchmark configurations): out = x + MoE(RMSNorm(x)).  RMSNorm has no
 * learned gain: xn = x / sqrt(mean(x^2) + 1e-6) per token, the sum of squares
 * in the router's fixed F32 order (coli_moe_dbg_rmsnorm runs it alone); the
 * residual add is fused into the combine (one F32 add after the weighted
 * sum).  The pre-norm is this library's reading: the pages chain the sweep's
 * layers with a residual add only, and without a norm the SwiGLU output grows
 * as the square of its input, so the stream overflows within a few layers.
 * Same arguments, rules and errors as coli_moe_layer_forward; `out` may not
 * alias `x`. */
int coli_moe_layer_forward_residual(const float *x, int n_tok,
                                    const float *router_w, const float *router_bias,
                                    const uint8_t *expert_w4, const float *expert_rowscale,
                                    const uint8_t *shared_w4, const float *shared_rowscale,
                                    float *out, void *stream);

/* coli_moe_layer_forward_residual with a layer-ahead prefetch for stacked
 * decode: while this layer's expert kernel finishes its last units, its
 * blocks that have run out of work pull the NEXT layer's router weights
 * (next_router_w, [E][H] F32) and shared expert (next_shared_w4, [3FH/2]
 * bytes) into L2.  Neither depends on the next layer's routing (the pages'
 * engine reads ahead asynchronously and reports router choices largely
 * predictable one layer ahead: "Colibri: an AI engine running a 744B model in
 * 25GB of RAM" (alphamatch.ai), section "Real performance"; only this
 * routing-independent part is prefetched here).  Results are identical to
 * coli_moe_layer_forward_residual.  Either next pointer may be NULL (nothing
 * of it is prefetched); both must be 16-byte aligned device pointers.  The
 * prefetch runs on the streaming path only (a prefill-sized batch takes the
 * grouped GEMM, which ignores them). */
int coli_moe_layer_forward_residual_prefetch(const float *x, int n_tok,
                                             const float *router_w, const float *router_bias,
                                             const uint8_t *expert_w4, const float *expert_rowscale,
                                             const uint8_t *shared_w4, const float *shared_rowscale,
                                             const float *next_router_w, const uint8_t *next_shared_w4,
                                             float *out, void *stream);

/* The same forward with x and out in HOST memory (pinned memory gives
 * asynchronous copies).  Copies x into a library-owned device buffer, runs the
 * forward and synchronises `stream` before returning, so out_host is valid on
 * return.  When out_host is page-locked and mapped into the device's address
 * space (cudaHostAlloc / cudaMallocHost memory, 16-byte aligned) the final
 * combine writes the result directly into it; any other host buffer receives
 * a copy of a library-owned device result.  Weights are device pointers. */
int coli_moe_layer_forward_hostio(const float *x_host, int n_tok,
                                  const float *router_w, const float *router_bias,
                                  const uint8_t *expert_w4, const float *expert_rowscale,
                                  const uint8_t *shared_w4, const float *shared_rowscale,
                                  float *out_host, void *stream);

/* Choose the expert-matmul path for later forwards (default COLI_PATH_AUTO).
 * `gemm_min_tokens`: with COLI_PATH_AUTO, a forward of at least this many
 * tokens runs the grouped tensor-core GEMM (the batch union of all experts:
 * gather of the activation codes by dispatch position, gate/up GEMM with
 * SiLU*up and Q8_0 of h, down GEMM, combine), a smaller one the streaming GEMV
 * kernel.  <= 0 keeps the built-in threshold: n_tok * top_k >=
 * COLI_GEMM_MIN_PAIRS_PER_EXPERT * n_experts, i.e. an average of 7 routed
 * tokens per expert (224 tokens for 256 experts top-8; measured crossover on
 * that shape between 192 and 256).  Returns COLI_E_INVAL for an unknown path.
 * Takes effect at the next forward; a forward with COLI_PATH_GEMM on a shape
 * whose ffn % 128 != 0 returns COLI_E_UNIMPL. */
#define COLI_GEMM_MIN_PAIRS_PER_EXPERT 7
int coli_moe_set_path(int path, int gemm_min_tokens);

/* Synchronise `stream`, then read and clear the device status word.
 * Returns COLI_OK, COLI_E_DEVICE (bad expert index seen), COLI_E_TIMEOUT
 * (a bounded device wait gave up) or COLI_E_CUDA. */
int coli_moe_get_device_status(void *stream);

/* Static, human-readable text for a status code. */
const char *coli_moe_strerror(int code);

/* Free the workspace and forget the shape.  Synchronises the device. */
void coli_moe_release(void);

/* Converter: quantise F32 weight rows to the int4 container, on the GPU.
 *   w [rows][K] F32 (K % 32 == 0) -> packed [rows][K/2], scale [rows] F32,
 * s = max|row| / 7 (IEEE divide), q = clamp(lrintf(w / s), -7, 7), nibble q+8,
 * low nibble first; an all-zero row gives s = 0 and codes 0 (model card
 * "GLM-5.2-colibri-int4", sections "TL;DR" and "Technical features").
 * Independent of coli_moe_configure(). */
int coli_moe_pack_int4(const float *w, int rows, int K, uint8_t *packed, float *scale,
                       void *stream);

/* The int8 weight container, on the GPU: w [rows][K] F32 (K % 32 == 0) ->
 * q [rows][K] int8 codes, scale [rows] F32, s = max|row| / 127 (IEEE
 * divide), q = clamp(lrintf(w / s), -127, 127); an all-zero row gives s = 0
 * and codes 0.  The int4 container's rule with 127 in place of 7: the pages
 * name an int8 container (to which the int4 packing decodes bit-identically)
 * and an int8 MTP head ("colibri: a pure-C inference engine ..."
 * (discuss.pytorch.kr), section "Key features"; "Open-source engine that ran
 * 744B GLM-5.2 ..." (jeff.news), section "MTP is sensitive").  One expert in
 * this container is gate [F][H], up [F][H], down [H][F] int8 codes back to
 * back (3*F*H bytes) with the same row scales [2F+H].  Independent of
 * coli_moe_configure(). */
int coli_moe_pack_int8(const float *w, int rows, int K, int8_t *q, float *scale, void *stream);

/* Weight container of later forwards: 4 (packed int4, the default) or 8 (the
 * int8 container of coli_moe_pack_int8; expert_w4 / shared_w4 then point at
 * 3*F*H bytes per expert).  Everything else is unchanged: Q8_0 activations,
 * int32 block dots, the same F32 fold and combine, on both expert paths.
 * Returns COLI_E_INVAL for other values. */
int coli_moe_set_weight_bits(int bits);

/* Kernel timing for measurement: when enabled, the library records CUDA events
 * around its dominant kernel (the expert gate/up + down matmuls) on the
 * forward's stream.  coli_moe_timing_read() synchronises, returns the summed
 * elapsed milliseconds and the number of timed launches, and resets them. */
int coli_moe_timing_enable(int on);
int coli_moe_timing_read(double *ms_total, int *n_timed);

/* Device-side event log of the expert kernel (tracing; off by default).
 * coli_moe_trace_enable(n) allocates a log of n events per block (n <= 4096;
 * 0 frees it and turns tracing off).  Each block writes, from its first
 * consumer thread, events (globaltimer_ns << 8 | code, unit): 1 kernel start,
 * 2 unit start, 3 activations staged, 4 unit done, 5 combine done, 6 exit;
 * word 0 of a block's log counts its events.  coli_moe_trace_read()
 * synchronises the device, copies the whole log (blocks x n x 2 u64) into
 * `host` (capacity in u64 elements), clears it, and reports its shape. */
int coli_moe_trace_enable(int events_per_block);
int coli_moe_trace_read(unsigned long long *host, long long capacity, int *blocks,
                        int *events_per_block);

/* Number of kernels the library launched since the last call (then reset). */
long long coli_moe_launch_count(void);

/* ---- host-memory expert tier -------------------------------------------------
 * The pages keep the dense weights in RAM and stream the routed experts from
 * disk on demand into RAM caches ("colibri: a pure-C inference engine ..."
 * (discuss.pytorch.kr), section "Core idea: dense in RAM, experts on disk";
 * "Open-source engine that ran 744B GLM-5.2 ..." (jeff.news), section
 * "Bottleneck: disk and RAM cache").  This tier is the same idea one level up:
 * the routed experts live in host memory (page-locked memory, read over the
 * host link: NVLink-C2C on a Grace host), and an LRU cache of them lives in a
 * pool of HBM slots.  Each forward routes on the GPU, brings the forward's
 * chosen experts to the host, copies every one that is not resident into the
 * least recently used slot not taken by this forward, and runs the expert
 * kernels on the slots.  The shared expert and the router stay in HBM.
 *
 * coli_moe_tier_configure(n_slots): after coli_moe_configure() (and
 *   coli_moe_set_weight_bits()): allocate n_slots HBM expert slots
 *   (1 <= n_slots <= n_experts; replaces an earlier tier).  COLI_E_NOMEM if
 *   the pool cannot be allocated.  coli_moe_configure() and
 *   coli_moe_release() free the tier.
 * coli_moe_tier_forward(): coli_moe_layer_forward's arguments, with the
 *   routed experts' weights and row scales in HOST memory:
 *   host_expert_w [E][3FH*bits/8], host_expert_rowscale [E][2F+H]
 *   (page-locked memory gives asynchronous copies).  Synchronises `stream`
 *   once, after routing, to read the choices; the expert launches follow
 *   asynchronously.  COLI_E_INVAL if one forward's union of experts exceeds
 *   the slots (before any copy or expert launch), or if the weight bits
 *   changed since the tier was configured.  Results are identical to
 *   coli_moe_layer_forward with the same weights in HBM.
 * coli_moe_tier_stats(): cumulative hits and misses (experts found resident
 *   or copied in), bytes copied to HBM, and the number of resident experts
 *   (any pointer may be NULL).
 * coli_moe_tier_release(): free the pool. */
int coli_moe_tier_configure(int n_slots);
int coli_moe_tier_forward(const float *x, int n_tok, const float *router_w, const float *router_bias,
                          const uint8_t *host_expert_w, const float *host_expert_rowscale,
                          const uint8_t *shared_w4, const float *shared_rowscale, float *out, void *stream);
int coli_moe_tier_stats(long long *hits, long long *misses, long long *bytes_h2d, int *resident);
void coli_moe_tier_release(void);

/* ---- routing without any device allocation --------------------------------
 * This entry point has no counterpart in the colibri pages: it is a service
 * for callers that must not allocate device memory (code running under
 * another runtime's allocator or memory pool, processes whose device memory is
 * fully reserved up front, serving loops that forbid allocation).  It runs
 * the same router as coli_moe_layer_forward (logits in the fixed F32 order,
 * sigmoid, +bias for selection, top-k with lowest-index ties, weights
 * sigma_r / sum(sigma_sel) * routed_scale) with the shape passed in `s`
 * (s->ffn and s->max_tok are ignored), and needs no coli_moe_configure().
 *   x [n_tok][H] F32 (16-byte aligned), router_w [E][H] F32 (16-byte
 *   aligned), router_bias [E] F32; outputs idx [n_tok][k] int32 (rank order)
 *   and w [n_tok][k] F32, all device pointers owned by the caller.
 * Its scratch (the logits) is a file-scope device array for at most
 * COLI_STATIC_MAX_TOK tokens and 256 experts, held on every GPU that loads the
 * library until exit; larger n_tok or E return COLI_E_INVAL.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current, so make that first call before any stream capture.  CUDA
 * loads module code and data lazily by default, so that first call is also
 * when the array's device memory is committed: make it before reserving the
 * rest of device memory (or set CUDA_MODULE_LOADING=EAGER).  The cached
 * address is invalid after cudaDeviceReset().  All calls share the one
 * array: calls that overlap on the GPU (different streams, or different host
 * threads) race on it. */
#define COLI_STATIC_MAX_TOK 64
int coli_moe_route_noalloc(const coli_moe_shape *s, const float *x, int n_tok,
                           const float *router_w, const float *router_bias, int32_t *idx, float *w,
                           void *stream);

/* ---- failure injection (tests) -------------------------------------------
 * Makes the library's own failure paths run without faulting or hanging the
 * GPU: every injected failure is decided on the host, or is a device-side wait
 * with a short bound that a test makes run out.  The pages' engine guards its
 * own resources the same way (it sizes its caches from MemAvailable so that
 * it never runs out of memory: "colibri: a pure-C inference engine ..."
 * (discuss.pytorch.kr), section "Core idea"); this library reports each
 * failure as a status and stays usable afterwards.
 *   COLI_INJECT_NONE          clear every injection (arg ignored)
 *   COLI_INJECT_ALLOC_FAIL    the next `arg` workspace allocations of
 *                             coli_moe_configure fail as if cudaMalloc had:
 *                             it returns COLI_E_NOMEM and leaves the library
 *                             unconfigured (no cudaMalloc is called)
 *   COLI_INJECT_LAUNCH_FAIL   the `arg`-th kernel launch from now (1 = the
 *                             next) is skipped and reported as a launch
 *                             failure: the call returns COLI_E_CUDA
 *   COLI_INJECT_WAIT_TIMEOUT  in the next streaming-path forward every down
 *                             unit waits for one more gate/up unit than its
 *                             tile has, with a bound of `arg` microseconds
 *                             instead of 2 s: each wait runs out, the
 *                             forward completes, and
 *                             coli_moe_get_device_status() then returns
 *                             COLI_E_TIMEOUT
 *   COLI_INJECT_GUARD         one byte of workspace guard region `arg`
 *                             (0 <= arg < the count coli_moe_dbg_check_guards
 *                             reports) is overwritten from the host, as a
 *                             stray device write past a buffer's end would
 *                             overwrite it; synchronises the device
 * 0 <= arg <= 1000000.  Returns COLI_E_INVAL for an unknown kind or an arg out
 * of range, COLI_E_NOSHAPE for COLI_INJECT_GUARD before configure. */
#define COLI_INJECT_NONE 0
#define COLI_INJECT_ALLOC_FAIL 1
#define COLI_INJECT_LAUNCH_FAIL 2
#define COLI_INJECT_WAIT_TIMEOUT 3
#define COLI_INJECT_GUARD 4
int coli_moe_dbg_inject(int what, long long arg);

/* ---- workspace guards (bounds checking without a sanitizer) ----------------
 * coli_moe_configure leaves a guard region between consecutive buffers of its
 * workspace (from each buffer's last byte at the configured maximum sizes to
 * the next buffer, at least 256 bytes) and 256 bytes before the first, filled
 * with the byte 0xA5.  No kernel writes there, so a guard that changed means
 * a write past a buffer's end.  This call synchronises the device, reads
 * every guard region back, restores the changed ones, and returns how many
 * had changed (0: all intact), or a negative coli_status (COLI_E_NOSHAPE
 * before configure, COLI_E_CUDA).  `n_guards` (optional) receives the number
 * of guard regions. */
int coli_moe_dbg_check_guards(int *n_guards);

/* ---- stage entry points (tests; same conventions, configured shape) ------- */

/* Q8_0 of n floats (n % 32 == 0): q [n] int8, d [n/32] F32 (same rule as the
 * forward's activation quantiser).  Independent of coli_moe_configure(). */
int coli_moe_dbg_quantize(const float *x, int n, int8_t *q, float *d, void *stream);

/* Router only: idx [n_tok][k] int32 (rank order), w [n_tok][k] F32;
 * optional logits [n_tok][E] F32 (NULL to skip). */
int coli_moe_dbg_route(const float *x, int n_tok, const float *router_w,
                       const float *router_bias, int32_t *idx, float *w, float *logits,
                       void *stream);

/* Stage entry point: the stacked layer's pre-norm alone.  x and xn [n_tok][hidden]
 * F32 device pointers (16-byte aligned, hidden % 4 == 0); needs no configure. */
int coli_moe_dbg_rmsnorm(const float *x, int n_tok, int hidden, float *xn, void *stream);

/* Dispatch only: from idx [n_tok][k] (values < E) produce counts [E],
 * offsets [E+1], perm [n_tok*k] (perm[pos] = pair t*k+r), inv [n_tok*k]. */
int coli_moe_dbg_dispatch(const int32_t *idx, int n_tok, int32_t *counts, int32_t *offsets,
                          int32_t *perm, int32_t *inv, void *stream);

/* Per-block int32 dot products of `rows` packed int4 rows of length K
 * (K % 32 == 0) with one int8 vector q [K]: I_out [rows][K/32]. */
int coli_moe_dbg_block_dots(const uint8_t *w4, int rows, int K, const int8_t *q,
                            int32_t *I_out, void *stream);

/* The same for rows of the int8 container: w8 [rows][K] int8 codes. */
int coli_moe_dbg_block_dots_w8(const int8_t *w8, int rows, int K, const int8_t *q, int32_t *I_out,
                               void *stream);

/* Measurement reference (needs no configure): one launch that streams `bytes`
 * bytes of the device buffer `buf` from HBM through bulk copies of `chunk`
 * bytes into per-block shared-memory rings of `stages` chunks, with
 * `blocks_per_sm` blocks per SM, each block a contiguous range, and does no
 * arithmetic on the data but a checksum: *sum (a device u64, zeroed by the
 * call) receives the sum of the four 32-bit words at every offset o < bytes
 * with o % 1024 == 0.  0 for chunk, stages or blocks_per_sm takes the one-token
 * expert kernel's arrangement (16384, 3, 4).  Limits: chunk 1024..65536 in steps of
 * 1024, stages 2..16, chunk * stages <= 200 KB, blocks_per_sm >= 1 and all
 * blocks resident; buf 16-byte aligned, bytes % 16 == 0, sum 8-byte aligned;
 * otherwise COLI_E_INVAL.  Its duration is the single-pass read time of that
 * many bytes, the floor against which the streaming expert kernel's
 * bandwidth is read. */
int coli_moe_dbg_stream_read(const void *buf, size_t bytes, int chunk, int stages, int blocks_per_sm,
                             unsigned long long *sum, void *stream);

/* Run a full forward and copy out its intermediates (any pointer may be NULL):
 * qx [n_tok][H] int8, dx [n_tok][H/32], idx/w [n_tok][k],
 * qh [n_tok*k + n_tok][F] int8 and dh [n_tok*k + n_tok][F/32] in pair order
 * (pair t*k+r, then the shared expert's rows t = 0..n_tok-1),
 * y [n_tok*k + n_tok][H] F32 per pair in the same order. */
int coli_moe_dbg_forward_intermediates(const float *x, int n_tok,
                                       const float *router_w, const float *router_bias,
                                       const uint8_t *expert_w4, const float *expert_rowscale,
                                       const uint8_t *shared_w4, const float *shared_rowscale,
                                       float *out, int8_t *qx, float *dx, int32_t *idx,
                                       float *w, int8_t *qh, float *dh, float *y,
                                       void *stream);

/* Gate/up + SiLU*up + Q8_0 of h for one expert on given quantized activations
 * (stage-isolated): qx [n][H] int8, dx [n][H/32] -> h [n][F] F32 (before
 * requantisation), qh [n][F] int8, dh [n][F/32].  1 <= n <= max_tok. */
int coli_moe_dbg_expert_hidden(const uint8_t *ew4, const float *ers, const int8_t *qx,
                               const float *dx, int n, float *h, int8_t *qh, float *dh,
                               void *stream);

#ifdef __cplusplus
}
#endif

#endif /* COLI_MOE_H */
