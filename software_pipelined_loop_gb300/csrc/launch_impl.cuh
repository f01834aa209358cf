// launch_impl.cuh -- launcher template shared by the kernel translation units.
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"
#include "variants.h"

namespace gp {

template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c, const GemmParams &p, int grid,
                       cudaStream_t s)
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
        if constexpr (Cfg::REG_SPLIT) {
            // setmaxnreg.inc waits until the CTA's launch allocation can
            // cover the warpgroups' new shares: refuse a build whose
            // allocation is smaller instead of launching a kernel that
            // would wait forever.
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, gemm_pipelined_kernel<Cfg>);
            if (e != cudaSuccess) return e;
            if (fa.numRegs * Cfg::THREADS < Cfg::SPLIT_REGS) return cudaErrorInvalidConfiguration;
        }
        attr_done[dev].store(1);
    }
    // Programmatic dependent launch: the CTAs may start (and run the set-up
    // that reads no global memory) while the previous grid finishes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (Cfg::PAIR) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = Cfg::CLUSTER;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    e = cudaLaunchKernelEx(&cfg, gemm_pipelined_kernel<Cfg>, a, b, c, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Number of clusters (CTA pairs, or quads of two pairs) of this variant the
// current device can hold at once (0 on error or for single-CTA variants).
template <class Cfg>
int max_pairs_cfg()
{
    if constexpr (!Cfg::PAIR) {
        return 0;
    } else {
        static std::atomic<int> cache[128];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
            cudaGetLastError();
            return 0;
        }
        int n = cache[dev].load();
        if (n > 0) return n;
        if (cudaFuncSetAttribute(gemm_pipelined_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaLaunchConfig_t cfg = {};
        constexpr int C = Cfg::CLUSTER;
        cfg.gridDim = dim3(C * (sms / C > 0 ? sms / C : 1), 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_pipelined_kernel<Cfg>, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return 0;
        }
        cache[dev].store(n);
        return n;
    }
}

template <class Cfg>
constexpr Variant make_variant()
{
    return Variant{{Cfg::LDG ? 1 : 0, Cfg::INT_OUT ? 1 : 0, Cfg::CONVERT ? 1 : 0, Cfg::BM, Cfg::BN, Cfg::BK,
                    Cfg::STAGES, Cfg::I8_STAGES, Cfg::QUAD ? 2 : (Cfg::PAIR ? 1 : 0), Cfg::THREADS, Cfg::SMEM_BYTES,
                    Cfg::SUM_IN_C ? 0 : 1, Cfg::TRACE ? 1 : 0},
                   &launch_cfg<Cfg>, &max_pairs_cfg<Cfg>};
}

}  // namespace gp
