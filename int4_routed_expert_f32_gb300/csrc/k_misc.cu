// k_misc.cu -- small helpers: tile-count bound and the stage-test gather of
// per-position rows into pair order.
#include "coli_common.cuh"
#include "coli_internal.h"

namespace coli {

int max_gemv_tiles(int T, int k, int E)
{
    const long P = (long)T * k;
    const long routed = P / GEMV_MT + (P < E ? P : E) + 1;
    return (int)(routed + (T + GEMV_MT - 1) / GEMV_MT);
}

// Copy per-position rows into pair order (pair p reads position inv[p]; the
// shared rows P + t stay where they are).
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
