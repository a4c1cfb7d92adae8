// stream_bench.cu -- read-only HBM streaming microbenchmark (minfer README
// M15: bench/roofline.cu, one launch streaming a large buffer with several
// 16-byte loads in flight per thread).  It measures what the GEMV kernel's
// access pattern can reach with no arithmetic: per-warp rings of 1-D bulk
// copies into shared memory (method 0), or 128-bit global loads (method 1).
#include "qgemv_launch.h"

namespace qg {

__global__ void stream_tma_kernel(const uint8_t *__restrict__ src, long long bytes, int stage_bytes, int D,
                                  unsigned long long *out, unsigned *status)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem) + warp * D;
    uint8_t *ring = smem + 128 * ((nw * D * 8 + 127) / 128) + static_cast<size_t>(warp) * D * stage_bytes;
    if (threadIdx.x == 0) s_abort = 0;
    if (lane == 0)
        for (int d = 0; d < D; ++d) mbar_init(&bar[d], 1);
    fence_mbar_init();
    __syncthreads();
    const long long nstages = bytes / stage_bytes;
    const long long s0 = nstages * blockIdx.x / gridDim.x, s1 = nstages * (blockIdx.x + 1) / gridDim.x;
    const uint64_t pol = l2_policy_evict_first();
    long long next = s0 + warp;  // stages of this warp: s0 + warp, + nw, ...
    int issued = 0;
    for (int d = 0; d < D && next < s1; ++d, next += nw, ++issued) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[d], stage_bytes);
            bulk_g2s(ring + d * stage_bytes, src + next * stage_bytes, stage_bytes, &bar[d], pol);
        }
    }
    unsigned long long acc = 0;
    int slot = 0;
    unsigned phase = 0;
    for (int c = 0; c < issued;) {
        if (!mbar_wait_bounded(&bar[slot], phase, &s_abort, status, WAIT_LIMIT_NS)) break;
        const uint4 v = *reinterpret_cast<const uint4 *>(ring + slot * stage_bytes + (lane * 16) % stage_bytes);
        acc ^= (static_cast<unsigned long long>(v.x) << 32) ^ v.w;
        __syncwarp();
        if (next < s1) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bar[slot], stage_bytes);
                bulk_g2s(ring + slot * stage_bytes, src + next * stage_bytes, stage_bytes, &bar[slot], pol);
            }
            next += nw;
            ++issued;
        }
        ++c;
        if (++slot == D) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (s_abort) {  // drain whatever is still in flight
        for (int d = 0; d < D; ++d) mbar_drain(&bar[d], 0), mbar_drain(&bar[d], 1);
    }
    if (acc == 0x9E3779B97F4A7C15ull) atomicXor(out, acc);  // keeps the loads live
}

template <int U>
__global__ void __launch_bounds__(512) stream_ldg_kernel(const uint4 *__restrict__ src, long long n16,
                                                         unsigned long long *out)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x * U;
    unsigned long long acc = 0;
    for (long long i = (static_cast<long long>(blockIdx.x) * blockDim.x) * U + threadIdx.x; i < n16; i += stride) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long k = i + static_cast<long long>(u) * blockDim.x;
            v[u] = k < n16 ? __ldcs(src + k) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) acc ^= (static_cast<unsigned long long>(v[u].x) << 32) ^ v[u].w;
    }
    if (acc == 0x9E3779B97F4A7C15ull) atomicXor(out, acc);
}

cudaError_t launch_stream_bench(const void *src, long long bytes, int method, int warps, int depth, int stage_bytes,
                                unsigned long long *out, unsigned *status, int sms, cudaStream_t st)
{
    if (method == 0) {
        const size_t smem = 128 * ((static_cast<size_t>(warps) * depth * 8 + 127) / 128) +
                            static_cast<size_t>(warps) * depth * stage_bytes;
        cudaError_t e = cudaFuncSetAttribute(stream_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        stream_tma_kernel<<<sms, warps * 32, smem, st>>>(static_cast<const uint8_t *>(src), bytes, stage_bytes, depth,
                                                         out, status);
    } else {
        const int threads = warps * 32;
        const long long n16 = bytes / 16;
        if (depth <= 4)
            stream_ldg_kernel<4><<<sms * 2, threads, 0, st>>>(static_cast<const uint4 *>(src), n16, out);
        else
            stream_ldg_kernel<8><<<sms * 2, threads, 0, st>>>(static_cast<const uint4 *>(src), n16, out);
    }
    return cudaGetLastError();
}

}  // namespace qg
