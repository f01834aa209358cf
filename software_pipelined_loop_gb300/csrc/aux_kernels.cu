// aux_kernels.cu -- the non-GEMM kernels of the library: int8 -> fp16
// widening of the INT8 path's operands, zero fill (K = 0), the streaming copy
// used as the in-run HBM reference, and the device status word.
#include <cuda_fp16.h>

#include <atomic>

#include "ptx.cuh"
#include "variants.h"

namespace gp {

__device__ int g_status_word;

// int8 -> fp16 for four packed bytes.  Biasing each byte by 128 gives
// u = v + 128 in [0, 255]; the fp16 bit pattern 0x6400 | u is 1024 + u
// exactly, and subtracting 1152 in fp16 leaves v exactly (integers below
// 2048 are representable).  Returns the halves of bytes 0,1 and 2,3.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

struct WidenJob {
    const int8_t *src;
    int64_t rows, cols;
    uint16_t *dst;
    int64_t pitch;  // destination row pitch in elements, a multiple of 8
};

// Loads the 16 int8 of one piece of row r (one 16-byte load when the row
// is 16-byte aligned and the piece whole, else byte loads of the valid ones).
__device__ __forceinline__ uint4 widen_load(const WidenJob &j, int64_t r, int64_t c)
{
    const int8_t *src = j.src + r * j.cols + c;
    const int64_t valid = j.cols - c;
    if (valid >= 16 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0)
        return __ldg(reinterpret_cast<const uint4 *>(src));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t x = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (4 * q + b < valid) x |= static_cast<uint32_t>(static_cast<uint8_t>(src[4 * q + b])) << (8 * b);
        w[q] = x;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Widens a loaded piece and writes its 16 fp16 values (slots past `cols` as
// zero: their bytes were loaded as 0, which widens to 0, and the mask keeps
// that independent of the load path).
__device__ __forceinline__ void widen_store(const WidenJob &j, int64_t r, int64_t c, const uint4 &v)
{
    uint32_t o[8];
    widen4(v.x, o[0], o[1]);
    widen4(v.y, o[2], o[3]);
    widen4(v.z, o[4], o[5]);
    widen4(v.w, o[6], o[7]);
    const int64_t valid = j.cols - c;
    if (valid < 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t e = 2 * q;
            const uint32_t keep = (e < valid ? 0x0000FFFFu : 0u) | (e + 1 < valid ? 0xFFFF0000u : 0u);
            o[q] &= keep;
        }
    }
    uint16_t *dst = j.dst + r * j.pitch + c;
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
    if (j.pitch - c > 8) reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// blockIdx.z picks the matrix (0: A, 1: B); x covers 16-element pieces of a
// row, y strides over rows.  Four rows' loads are issued before any of them
// is widened and stored, so each thread keeps four loads in flight.
__global__ void widen_s8_f16_kernel(const WidenJob ja, const WidenJob jb)
{
    const WidenJob &j = blockIdx.z == 0 ? ja : jb;
    const int64_t c = 16 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (c >= j.pitch) return;
    const int64_t step = gridDim.y;
    int64_t r = blockIdx.y;
    for (; r + 3 * step < j.rows; r += 4 * step) {
        const uint4 v0 = widen_load(j, r, c);
        const uint4 v1 = widen_load(j, r + step, c);
        const uint4 v2 = widen_load(j, r + 2 * step, c);
        const uint4 v3 = widen_load(j, r + 3 * step, c);
        widen_store(j, r, c, v0);
        widen_store(j, r + step, c, v1);
        widen_store(j, r + 2 * step, c, v2);
        widen_store(j, r + 3 * step, c, v3);
    }
    for (; r < j.rows; r += step) widen_store(j, r, c, widen_load(j, r, c));
}

// Copies a rows x cols fp16 matrix (densely packed, any 2-byte alignment)
// into a destination whose row pitch `pitch` is a multiple of 8 elements,
// the slots past `cols` set to zero.  Each thread writes 8 elements (16
// bytes) of a row: it reads the two naturally aligned 16-byte words that
// hold them -- each is read only if it contains a byte of the row, so no
// read leaves the source allocation -- and shifts them into place.
struct PadJob {
    const uint16_t *src;
    int64_t rows, cols;
    uint16_t *dst;
    int64_t pitch;
};

struct PadLoad {
    uint4 w0, w1;
    uint32_t s;
};

__device__ __forceinline__ PadLoad pad_load(const PadJob &j, int64_t r, int64_t c)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(j.src + r * j.cols);
    const uintptr_t hi = lo + 2 * static_cast<uintptr_t>(j.cols);
    const uintptr_t a = lo + 2 * static_cast<uintptr_t>(c);
    PadLoad L;
    L.s = static_cast<uint32_t>(a & 15u);
    const uintptr_t base = a - L.s;
    L.w0 = make_uint4(0, 0, 0, 0);
    L.w1 = make_uint4(0, 0, 0, 0);
    if (base < hi && base + 16 > lo) L.w0 = __ldg(reinterpret_cast<const uint4 *>(base));
    if (L.s != 0 && base + 16 < hi) L.w1 = __ldg(reinterpret_cast<const uint4 *>(base + 16));
    return L;
}

__device__ __forceinline__ void pad_store(const PadJob &j, int64_t r, int64_t c, const PadLoad &L)
{
    uint32_t o[4];
    realign16(L.w0, L.w1, L.s, o);
    const int64_t valid = j.cols - c;
    if (valid < 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t keep = (2 * i < valid ? 0x0000FFFFu : 0u) | (2 * i + 1 < valid ? 0xFFFF0000u : 0u);
            o[i] &= keep;
        }
    }
    *reinterpret_cast<uint4 *>(j.dst + r * j.pitch + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

// x covers 8-element pieces of a row, y strides over rows with four rows'
// loads in flight per thread; z picks one of two jobs (A and B padded in
// one launch).
__global__ void pad_f16_kernel(const PadJob j0, const PadJob j1)
{
    const PadJob &j = blockIdx.z == 0 ? j0 : j1;
    const int64_t c = 8 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (c >= j.pitch) return;
    const int64_t step = gridDim.y;
    int64_t r = blockIdx.y;
    for (; r + 3 * step < j.rows; r += 4 * step) {
        const PadLoad l0 = pad_load(j, r, c);
        const PadLoad l1 = pad_load(j, r + step, c);
        const PadLoad l2 = pad_load(j, r + 2 * step, c);
        const PadLoad l3 = pad_load(j, r + 3 * step, c);
        pad_store(j, r, c, l0);
        pad_store(j, r + step, c, l1);
        pad_store(j, r + 2 * step, c, l2);
        pad_store(j, r + 3 * step, c, l3);
    }
    for (; r < j.rows; r += step) pad_store(j, r, c, pad_load(j, r, c));
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
    const WidenJob ja{A, rowsA, colsA, A16, pitchA};
    const WidenJob jb{B, rowsB, colsB, B16, pitchB};
    const int threads = 128;
    const int64_t maxpitch = pitchA > pitchB ? pitchA : pitchB;
    const int64_t gx = ((maxpitch + 15) / 16 + threads - 1) / threads;
    const int64_t maxrows = rowsA > rowsB ? rowsA : rowsB;
    // About eight blocks of 128 threads per SM for each matrix.
    int64_t gy = (static_cast<int64_t>(sms) * 8 + gx - 1) / gx;
    // Prefer whole groups of four rows per y-block.
    if (gy * 4 > maxrows) gy = (maxrows + 3) / 4;
    gy = gy < 1 ? 1 : (gy > maxrows ? maxrows : gy);
    gy = gy > 65535 ? 65535 : gy;
    if (gx > 2147483647) return cudaErrorInvalidValue;
    widen_s8_f16_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 2), threads, 0, s>>>(ja, jb);
    return cudaGetLastError();
}

cudaError_t launch_pad_f16(const uint16_t *src0, int64_t rows0, int64_t cols0, uint16_t *dst0, int64_t pitch0,
                           const uint16_t *src1, int64_t rows1, int64_t cols1, uint16_t *dst1, int64_t pitch1,
                           int sms, cudaStream_t s)
{
    // rows1 == 0: one job only.
    const PadJob j0{src0, rows0, cols0, dst0, pitch0};
    const PadJob j1{src1, rows1, cols1, dst1, pitch1};
    const int threads = 128;
    const int64_t maxpitch = pitch0 > pitch1 ? pitch0 : pitch1;
    const int64_t maxrows = rows0 > rows1 ? rows0 : rows1;
    const int64_t gx = (maxpitch / 8 + threads - 1) / threads;
    int64_t gy = (static_cast<int64_t>(sms) * 16 + gx - 1) / gx;
    if (gy * 4 > maxrows) gy = (maxrows + 3) / 4;
    gy = gy < 1 ? 1 : (gy > maxrows ? maxrows : gy);
    gy = gy > 65535 ? 65535 : gy;
    if (gx > 2147483647) return cudaErrorInvalidValue;
    const unsigned gz = rows1 > 0 ? 2u : 1u;
    pad_f16_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), gz), threads, 0, s>>>(j0, j1);
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
