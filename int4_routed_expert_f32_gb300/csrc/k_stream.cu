// k_stream.cu -- a bare one-pass read of a device buffer, for measurement:
// the rate at which one launch can stream a given number of bytes from HBM
// through the same machinery the expert kernel uses (bulk copies into a
// per-block shared-memory ring, completion on mbarriers, a consumer warp that
// releases each stage), with no arithmetic on the data.  It is the reference
// the expert kernel's bandwidth is compared with: a single pass over ~170 MB
// is bounded by its ramp and tail, not only by the HBM copy rate measured on
// gigabyte buffers.
//
// Each block streams one contiguous range of chunks (one bulk copy each, a
// ring of `stages` of them); the consumer reads the first 16 bytes of every
// 1 KB of each chunk and adds their four 32-bit words into a 64-bit sum, so
// that the call's result can be checked on the host and the copies cannot be
// elided.  Chunk size, ring depth and blocks per SM are parameters, so that
// the same call sweeps the read's configurations.
#include <cuda.h>

#include "coli_common.cuh"
#include "coli_internal.h"
#include "tma.cuh"

namespace coli {

constexpr int S_MAX_STAGES = 16;
constexpr int S_THREADS = 64;       // warp 0 lane 0: producer; warp 1: consumer
constexpr uint64_t S_WAIT_NS = 2000000000ull;

__device__ __forceinline__ uint64_t s_timer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// 1-D bulk copy global -> shared completing on bar (both addresses 16-byte
// aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool s_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = s_timer();
    while (!mbar_try_wait(bar, parity))
        if (s_timer() - t0 > S_WAIT_NS) return false;
    return true;
}

__global__ void __launch_bounds__(S_THREADS)
k_stream_read(const unsigned char *__restrict__ buf, size_t bytes, int chunk, int stages, unsigned long long *sum,
              int *status)
{
    extern __shared__ __align__(128) unsigned char ring[];     // [stages][chunk]
    __shared__ __align__(8) uint64_t full[S_MAX_STAGES], empty[S_MAX_STAGES];
    __shared__ int abort_flag;
    const size_t n_chunks = (bytes + chunk - 1) / chunk;
    const size_t per = (n_chunks + gridDim.x - 1) / gridDim.x;
    const size_t c0 = (size_t)blockIdx.x * per;
    const size_t c1 = c0 + per < n_chunks ? c0 + per : n_chunks;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0) {
            for (size_t c = c0; c < c1; ++c) {
                const int i = (int)(c - c0), slot = i % stages;
                if (i >= stages && !s_wait(&empty[slot], (uint32_t)(((i / stages) - 1) & 1))) {
                    set_status(status, ST_TIMEOUT);
                    abort_flag = 1;
                    // complete the consumer's pending phase without data
                    mbar_arrive(&full[slot]);
                    break;
                }
                const size_t off = c * (size_t)chunk;
                const uint32_t n = (uint32_t)(bytes - off < (size_t)chunk ? bytes - off : (size_t)chunk);
                mbar_arrive_expect_tx(&full[slot], n);
                bulk_load(ring + (size_t)slot * chunk, buf + off, n, &full[slot]);
            }
        }
        return;
    }
    // consumer warp
    unsigned long long acc = 0;
    for (size_t c = c0; c < c1; ++c) {
        const int i = (int)(c - c0), slot = i % stages;
        if (!s_wait(&full[slot], (uint32_t)((i / stages) & 1))) {
            if (lane == 0) set_status(status, ST_TIMEOUT);
            break;
        }
        if (abort_flag) break;
        const size_t off = c * (size_t)chunk;
        const size_t n = bytes - off < (size_t)chunk ? bytes - off : (size_t)chunk;
        for (int o = lane * 1024; (size_t)o < n; o += 32 * 1024) {
            const uint4 v = *reinterpret_cast<const uint4 *>(ring + (size_t)slot * chunk + o);
            acc += (unsigned long long)v.x + v.y + v.z + v.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
    if (lane == 0) atomicAdd(sum, acc);
}

int launch_stream_read(const void *buf, size_t bytes, int chunk, int stages, int blocks_per_sm,
                       unsigned long long *sum, int *status, int num_sms, cudaStream_t st)
{
    if (bytes == 0) return 0;
    const int smem = chunk * stages;
    static int configured = 0;
    if (smem > configured) {
        if (cudaFuncSetAttribute(k_stream_read, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return -1;
        configured = smem;
    }
    k_stream_read<<<num_sms * blocks_per_sm, S_THREADS, smem, st>>>(static_cast<const unsigned char *>(buf), bytes,
                                                                      chunk, stages, sum, status);
    count_launch();
    return 0;
}

}  // namespace coli
