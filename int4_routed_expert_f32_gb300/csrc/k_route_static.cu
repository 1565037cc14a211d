// k_route_static.cu -- the router (logits, sigmoid, top-k, renormalised
// weights) for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code running inside another
// runtime's memory pool or allocator hooks, in a process whose device memory
// is fully pre-reserved, or in a capture-sensitive serving loop that must not
// trigger allocation.  For them this entry point keeps its scratch (the router
// logits) in a file-scope __device__ array, so it needs no workspace and no
// prior coli_moe_configure() call.  The array is sized for at most
// COLI_STATIC_MAX_TOK tokens and 256 experts and stays resident on every GPU
// that loads this library until the process exits.
#include <atomic>
#include <cstdio>

#include "../../include/coli_moe.h"
#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

constexpr int STATIC_MAX_TOK = COLI_STATIC_MAX_TOK;
constexpr int STATIC_MAX_E = 256;
constexpr int MAX_DEVICES = 64;

// Router logits of the last call: [n_tok][E] F32.  Every call overwrites the
// region it reads, so nothing has to start at zero.
static __device__ __align__(256) float g_static_logits[STATIC_MAX_TOK * STATIC_MAX_E];

// Device address of g_static_logits per device.  In host code the array's
// name is a host-side stand-in, not a device address, so the address is
// looked up once per device (with that device current) and cached.  The
// entries are atomics: two host threads making their first call on the same
// device look up the same address, and either store is correct.  A cached
// address belongs to the device's current context: after cudaDeviceReset()
// it is stale, and the library must be reloaded before this call is used
// again on that device.
//
// CUDA loads a module's device code and data lazily by default, so the first
// call on a device (the symbol lookup or the first launch) is when the
// array's device memory is committed.  A caller that reserves all remaining
// device memory, or captures streams, should make one call first (or run
// with CUDA_MODULE_LOADING=EAGER).
static std::atomic<float *> g_static_logits_dev[MAX_DEVICES];

static int static_scratch(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        (void)cudaGetLastError();
        return COLI_E_CUDA;
    }
    float *p = g_static_logits_dev[dev].load(std::memory_order_acquire);
    if (!p) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_static_logits) != cudaSuccess || !a) {
            (void)cudaGetLastError();
            return COLI_E_CUDA;
        }
        p = static_cast<float *>(a);
        g_static_logits_dev[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return COLI_OK;
}

}  // namespace coli

using namespace coli;

extern "C" int coli_moe_route_noalloc(const coli_moe_shape *s, const float *x, int n_tok,
                                      const float *router_w, const float *router_bias, int32_t *idx,
                                      float *w, void *stream)
{
    if (!s) return COLI_E_INVAL;
    if (s->hidden <= 0 || s->hidden % 128 != 0 || s->hidden > 16384) return COLI_E_INVAL;
    if (s->n_experts < 1 || s->n_experts > STATIC_MAX_E) return COLI_E_INVAL;
    if (s->top_k < 1 || s->top_k > 16 || s->top_k > s->n_experts) return COLI_E_INVAL;
    if (!(s->routed_scale > 0.0f) || s->routed_scale > 3.0e38f) return COLI_E_INVAL;
    if (n_tok < 0 || n_tok > STATIC_MAX_TOK) return COLI_E_INVAL;
    if (n_tok == 0) return COLI_OK;
    if (!x || !router_w || !router_bias || !idx || !w) return COLI_E_INVAL;
    if (((uintptr_t)x & 15u) || ((uintptr_t)router_w & 15u)) return COLI_E_INVAL;
    float *logits = nullptr;
    const int st = static_scratch(&logits);
    if (st != COLI_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    if (launch_router_logits(x, n_tok, s->hidden, router_w, s->n_experts, logits, cs) != 0 ||
        cudaGetLastError() != cudaSuccess)
        return COLI_E_CUDA;
    if (launch_topk(logits, n_tok, s->n_experts, s->top_k, router_bias, s->routed_scale, idx, w, cs) != 0 ||
        cudaGetLastError() != cudaSuccess)
        return COLI_E_CUDA;
    return COLI_OK;
}
