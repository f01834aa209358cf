// aux_kernels.cu -- the non-GEMM kernels of the library: int8 -> fp16
// widening of the INT8 path's operands, zero fill (K = 0), the streaming copy
// used as the in-run HBM reference, and the device status word.
#include <cuda_fp16.h>

#include <atomic>

#include "variants.h"

namespace gp {

__device__ int g_status_word;

// Widen one int8 row segment of up to 16 values into fp16 bit patterns.
__device__ __forceinline__ void widen16(const int8_t *src, int64_t valid, uint16_t *dst, int64_t room)
{
    uint16_t h[16];
    if (valid >= 16 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int8_t b = static_cast<int8_t>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
            h[i] = __half_as_ushort(__short2half_rn(static_cast<short>(b)));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            h[i] = i < valid ? __half_as_ushort(__short2half_rn(static_cast<short>(src[i]))) : 0;
    }
    // room: fp16 slots left in the destination row (a multiple of 8)
    uint4 o0, o1;
    o0.x = h[0] | (uint32_t(h[1]) << 16);
    o0.y = h[2] | (uint32_t(h[3]) << 16);
    o0.z = h[4] | (uint32_t(h[5]) << 16);
    o0.w = h[6] | (uint32_t(h[7]) << 16);
    o1.x = h[8] | (uint32_t(h[9]) << 16);
    o1.y = h[10] | (uint32_t(h[11]) << 16);
    o1.z = h[12] | (uint32_t(h[13]) << 16);
    o1.w = h[14] | (uint32_t(h[15]) << 16);
    reinterpret_cast<uint4 *>(dst)[0] = o0;
    if (room > 8) reinterpret_cast<uint4 *>(dst)[1] = o1;
}

// Rows [0, rowsA) of the flattened row range belong to A, the rest to B.
// Each destination row has `pitch` (a multiple of 8) fp16 slots; the slots
// past the source columns are written as zero.
__global__ void widen_s8_f16_kernel(const int8_t *A, int64_t rowsA, int64_t colsA, uint16_t *A16,
                                    int64_t pitchA, const int8_t *B, int64_t rowsB, int64_t colsB,
                                    uint16_t *B16, int64_t pitchB)
{
    const int64_t rows = rowsA + rowsB;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const bool isA = r < rowsA;
        const int64_t row = isA ? r : r - rowsA;
        const int64_t cols = isA ? colsA : colsB;
        const int64_t pitch = isA ? pitchA : pitchB;
        const int8_t *src = (isA ? A : B) + row * cols;
        uint16_t *dst = (isA ? A16 : B16) + row * pitch;
        for (int64_t c = 16 * static_cast<int64_t>(threadIdx.x); c < pitch; c += 16 * blockDim.x)
            widen16(src + c, cols - c, dst + c, pitch - c);
    }
}

__global__ void zero_fill_kernel(uint8_t *dst, int64_t bytes)
{
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(dst);
    if ((addr & 15u) == 0) {
        const int64_t n16 = bytes / 16;
        for (int64_t i = tid; i < n16; i += nth) reinterpret_cast<uint4 *>(dst)[i] = make_uint4(0, 0, 0, 0);
        for (int64_t i = 16 * n16 + tid; i < bytes; i += nth) dst[i] = 0;
    } else {
        for (int64_t i = tid; i < bytes; i += nth) dst[i] = 0;
    }
}

__global__ void copy_kernel(uint8_t *dst, const uint8_t *src, int64_t bytes)
{
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0) {
        const int64_t n16 = bytes / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int64_t i = tid; i < n16; i += nth) d[i] = s[i];
        for (int64_t i = 16 * n16 + tid; i < bytes; i += nth) dst[i] = src[i];
    } else {
        for (int64_t i = tid; i < bytes; i += nth) dst[i] = src[i];
    }
}

cudaError_t launch_widen_s8_f16(const int8_t *A, int64_t rowsA, int64_t colsA, uint16_t *A16, int64_t pitchA,
                                const int8_t *B, int64_t rowsB, int64_t colsB, uint16_t *B16, int64_t pitchB,
                                int sms, cudaStream_t s)
{
    const int64_t rows = rowsA + rowsB;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int grid = static_cast<int>(rows < cap ? rows : cap);
    const int64_t maxpitch = pitchA > pitchB ? pitchA : pitchB;
    int threads = static_cast<int>((maxpitch + 15) / 16);
    threads = threads < 32 ? 32 : (threads > 256 ? 256 : (threads + 31) / 32 * 32);
    widen_s8_f16_kernel<<<grid, threads, 0, s>>>(A, rowsA, colsA, A16, pitchA, B, rowsB, colsB, B16, pitchB);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *dst, int64_t bytes, int sms, cudaStream_t s)
{
    const int64_t need = (bytes / 16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 4;
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    zero_fill_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t *>(dst), bytes);
    return cudaGetLastError();
}

cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, int sms, cudaStream_t s)
{
    const int64_t need = (bytes / 16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    copy_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t *>(dst), static_cast<const uint8_t *>(src), bytes);
    return cudaGetLastError();
}

cudaError_t status_word(int **ptr)
{
    static std::atomic<int *> cache[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    int *p = cache[dev].load();
    if (!p) {
        void *a = nullptr;
        e = cudaGetSymbolAddress(&a, g_status_word);
        if (e != cudaSuccess) return e;
        p = static_cast<int *>(a);
        cache[dev].store(p);
    }
    *ptr = p;
    return cudaSuccess;
}

}  // namespace gp
