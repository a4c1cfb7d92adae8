// launch_stream.cuh -- launcher of the streaming GEMV kernel; included by
// the per-T translation units, which instantiate it.
#pragma once

#include <atomic>

#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

namespace qg {

template <int T, int MAXG, bool ARGMAX, bool MMA, bool EPI>
cudaError_t launch_stream(const Params<MAXG> &P, int grid, size_t smem, cudaStream_t st, bool pdl)
{
    auto kern = qgemv_stream_kernel<T, MAXG, ARGMAX, MMA, EPI>;
    // The dynamic shared-memory limit is a per-device function attribute:
    // raise it once per device to the largest size any launch asks for.
    static std::atomic<unsigned long long> raised{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(raised.load(std::memory_order_acquire) & bit)) {
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(P.nwarps * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace qg
