// gemm_noalloc.cu -- gemm_s8s8s32_noalloc: the INT8 GEMM for callers that
// cannot let the library allocate device memory (see include/gemmpipe.h).
//
// The fp16 copies of the operands go into one fixed array declared here in
// device memory.  Host code must not use the array's name as an address (on
// the host it is only a stand-in, and a kernel given it would fault or
// silently use the wrong memory), so the device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, and
// passed to the kernels.
#include <cuda_runtime.h>

#include <atomic>

#include "gemmpipe.h"
#include "variants.h"

namespace {

constexpr int64_t kScratchBytes = GEMMPIPE_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; held from library load to process exit.
static __device__ __align__(256) uint16_t g_s8_scratch[kScratchBytes / 2];

std::atomic<uint16_t *> g_scratch_addr[128];

// Device address of g_s8_scratch on the current device (looked up on the
// first call made with that device current).  Under CUDA's lazy module
// loading that lookup is also what loads this file's device code on the
// device and so creates the array; a device without room for it gives
// GEMMPIPE_ERR_OUT_OF_MEMORY.
gemmpipe_status_t scratch_address(uint16_t **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
        cudaGetLastError();
        return GEMMPIPE_ERR_UNSUPPORTED_DEVICE;
    }
    uint16_t *p = g_scratch_addr[dev].load();
    if (!p) {
        void *a = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&a, g_s8_scratch);
        if (e != cudaSuccess || !a) {
            cudaGetLastError();
            return e == cudaErrorMemoryAllocation ? GEMMPIPE_ERR_OUT_OF_MEMORY : GEMMPIPE_ERR_LAUNCH;
        }
        p = static_cast<uint16_t *>(a);
        g_scratch_addr[dev].store(p);
    }
    *out = p;
    return GEMMPIPE_OK;
}

}  // namespace

extern "C" gemmpipe_status_t gemm_s8s8s32_noalloc(int64_t M, int64_t N, int64_t K, const int8_t *A,
                                                  const int8_t *B, int32_t *C, gemmpipe_stream_t stream)
{
    // Size and argument checks first: too-large problems are refused before
    // any device work or set-up.
    gemmpipe_status_t st = gp::s8_check_fixed_scratch(M, N, K, A, B, C, kScratchBytes);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    uint16_t *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != GEMMPIPE_OK) return st;
    return gp::s8_with_fixed_scratch(M, N, K, A, B, C, reinterpret_cast<cudaStream_t>(stream), scratch,
                                     kScratchBytes);
}
