// launch_impl.cuh -- launcher template shared by the kernel translation units.
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"
#include "variants.h"

namespace gp {

template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, int grid, cudaStream_t s)
{
    static std::atomic<int> attr_done[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!attr_done[dev].load()) {
        e = cudaFuncSetAttribute(gemm_pipelined_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev].store(1);
    }
    gemm_pipelined_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, s>>>(a, b, p);
    return cudaGetLastError();
}

template <class Cfg>
constexpr Variant make_variant()
{
    return Variant{{Cfg::LDG ? 1 : 0, Cfg::INT_OUT ? 1 : 0, Cfg::CONVERT ? 1 : 0, Cfg::BM, Cfg::BN, Cfg::BK,
                    Cfg::STAGES, Cfg::I8_STAGES, Cfg::THREADS, Cfg::SMEM_BYTES},
                   &launch_cfg<Cfg>};
}

}  // namespace gp
