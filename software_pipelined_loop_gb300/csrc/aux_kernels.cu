// aux_kernels.cu -- the non-GEMM kernels of the library: int8 -> fp16
// widening of the INT8 path's operands, zero fill (K = 0), the streaming copy
// used as the in-run HBM reference, and the device status word.
#include <cuda_fp16.h>

#include <atomic>
#include <utility>

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
    int64_t spitch;  // source row pitch in elements (>= cols)
    uint16_t *dst;
    int64_t pitch;  // destination row pitch in elements, a multiple of 8
    int64_t dcols;  // destination columns written (>= cols, a multiple of 8; past cols: zeros)
};

// Loads the 16 int8 of one piece of row r (one 16-byte load when the row
// is 16-byte aligned and the piece whole, else byte loads of the valid ones).
__device__ __forceinline__ uint4 widen_load(const WidenJob &j, int64_t r, int64_t c)
{
    const int8_t *src = j.src + r * j.spitch + c;
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
    if (j.dcols - c > 8) reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// blockIdx.z picks the matrix (0: A, 1: B); x covers 16-element pieces of a
// row, y strides over rows.  Each thread issues the loads of up to kRowBatch
// rows (its last batch predicated) before widening and storing any of them,
// so a thread's rows cost one memory round trip per batch.
constexpr int kRowBatch = 8;

__global__ void widen_s8_f16_kernel(const WidenJob ja, const WidenJob jb)
{
    pdl_wait();
    pdl_launch_dependents();
    const WidenJob &j = blockIdx.z == 0 ? ja : jb;
    const int64_t c = 16 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (c >= j.dcols) return;
    const int64_t step = gridDim.y;
    for (int64_t r = blockIdx.y; r < j.rows; r += kRowBatch * step) {
        uint4 v[kRowBatch];
#pragma unroll
        for (int i = 0; i < kRowBatch; ++i)
            if (r + i * step < j.rows) v[i] = widen_load(j, r + i * step, c);
#pragma unroll
        for (int i = 0; i < kRowBatch; ++i)
            if (r + i * step < j.rows) widen_store(j, r + i * step, c, v[i]);
    }
}

// Widening of operands whose rows are whole 16-byte units (cols a multiple
// of 16, 16-byte aligned bases, destination pitch == cols): each matrix is
// one contiguous array of n int8 (n a multiple of 16) and becomes n fp16.
// One CTA per SM streams 16 KiB chunks: a bulk copy brings a chunk into one
// of kFlatInStages shared-memory stages (completion on the stage's
// mbarrier), the threads widen it into one of kFlatOut output buffers, and
// a bulk copy writes that to global memory.  Loads run kFlatInStages chunks
// ahead; one CTA barrier per chunk orders the widening before the store.
struct FlatJob {
    const int8_t *src;
    uint16_t *dst;
    int64_t n;
};

constexpr int kFlatChunk = 16384;  // int8 bytes per chunk
constexpr int kFlatInStages = 6;
constexpr int kFlatOut = 3;
constexpr int kFlatThreads = 256;
constexpr int kFlatSmem = kFlatInStages * kFlatChunk + kFlatOut * 2 * kFlatChunk + 8 * kFlatInStages + 128;
static_assert(kFlatOut >= 3, "an output buffer is rewritten two chunks after its store was confirmed read");
// Bulk stores allowed to still read shared memory at the end of an
// iteration: the buffer of chunk i + 2 was last read by the store of chunk
// i + 2 - kFlatOut, which is then finished.
static_assert(kFlatSmem <= 232448, "over the per-CTA shared-memory limit");

__global__ void __launch_bounds__(kFlatThreads, 1)
    widen_flat_kernel(const FlatJob ja, const FlatJob jb, int *status, uint64_t timeout_ns)
{
    extern __shared__ __align__(128) uint8_t fsm[];
    const uint32_t base = (smem_u32(fsm) + 127u) & ~127u;
    const uint32_t in0 = base;
    const uint32_t out0 = base + kFlatInStages * kFlatChunk;
    const uint32_t bar0 = out0 + kFlatOut * 2 * kFlatChunk;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t ca = (ja.n + kFlatChunk - 1) / kFlatChunk;
    const int64_t total = ca + (jb.n + kFlatChunk - 1) / kFlatChunk;
    const int64_t mine = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    // Source, destination and size of this CTA's i-th chunk.
    auto chunk = [&](int64_t i, const int8_t *&src, uint16_t *&dst, uint32_t &bytes) {
        const int64_t g = blockIdx.x + i * gridDim.x;
        const FlatJob &j = g < ca ? ja : jb;
        const int64_t off = (g < ca ? g : g - ca) * kFlatChunk;
        const int64_t left = j.n - off;
        bytes = static_cast<uint32_t>(left < kFlatChunk ? left : kFlatChunk);
        src = j.src + off;
        dst = j.dst + off;
    };
    auto issue = [&](int64_t i) {
        const int8_t *src;
        uint16_t *dst;
        uint32_t bytes;
        chunk(i, src, dst, bytes);
        const int st = static_cast<int>(i % kFlatInStages);
        mbar_arrive_expect_tx(bar0 + 8 * st, bytes);
        bulk_load_g2s(in0 + st * kFlatChunk, src, bytes, bar0 + 8 * st);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < kFlatInStages; ++st) mbar_init(bar0 + 8 * st, 1);
        fence_mbar_init();
        for (int64_t i = 0; i < mine && i < kFlatInStages; ++i) issue(i);
    }
    __syncthreads();
    int64_t issued = mine < kFlatInStages ? mine : kFlatInStages;
    int64_t i = 0;
    for (; i < mine; ++i) {
        const int st = static_cast<int>(i % kFlatInStages);
        const uint32_t parity = static_cast<uint32_t>((i / kFlatInStages) & 1);
        const uint32_t ob = out0 + static_cast<uint32_t>(i % kFlatOut) * (2 * kFlatChunk);
        bool late = false;
        if (!mbar_try_wait(bar0 + 8 * st, parity)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar0 + 8 * st, parity))
                if (globaltimer_ns() - t0 > timeout_ns) {
                    late = true;
                    break;
                }
        }
        const int8_t *src;
        uint16_t *dst;
        uint32_t bytes;
        chunk(i, src, dst, bytes);
        if (!late) {
            // 8 int8 -> 8 fp16 per step; a warp reads 256 and writes 512
            // contiguous bytes.
            const uint32_t ib = in0 + st * kFlatChunk;
            for (uint32_t b = 8 * threadIdx.x; b < bytes; b += 8 * kFlatThreads) {
                const uint2 v = ld_shared_v2(ib + b);
                uint32_t o0, o1, o2, o3;
                widen4(v.x, o0, o1);
                widen4(v.y, o2, o3);
                st_shared_v4(ob + 2 * b, o0, o1, o2, o3);
            }
            fence_proxy_async_smem();
        }
        if (__syncthreads_or(late)) break;
        if (threadIdx.x == 0) {
            bulk_store_s2g(dst, ob, 2 * bytes);
            bulk_commit();
            if (issued < mine) {
                issue(issued);  // into stage st, just consumed
                ++issued;
            }
            // The output buffer of chunk i + 2 was last read by the store of
            // chunk i + 2 - kFlatOut: done once at most kFlatOut - 2 groups
            // (the newest stores) are still reading.
            bulk_wait_read<kFlatOut - 2>();
        }
    }
    if (threadIdx.x == 0) {
        if (i < mine) {
            // A load ran out of time: record it, and let every load still
            // in flight land before the CTA's shared memory goes away.
            atomicCAS(status, 0, static_cast<int>(GEMMPIPE_ERR_TIMEOUT));
            for (int64_t k = i; k < issued; ++k) {
                const int st = static_cast<int>(k % kFlatInStages);
                const uint32_t parity = static_cast<uint32_t>((k / kFlatInStages) & 1);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar0 + 8 * st, parity))
                    if (globaltimer_ns() - t0 > timeout_ns) break;
            }
        }
        bulk_wait<0>();
    }
    __syncthreads();
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

// x covers 8-element pieces of a row, y strides over rows in batches of
// kRowBatch rows whose loads are all in flight together; z picks one of two
// jobs (A and B padded in one launch).
__global__ void pad_f16_kernel(const PadJob j0, const PadJob j1)
{
    pdl_wait();
    pdl_launch_dependents();
    const PadJob &j = blockIdx.z == 0 ? j0 : j1;
    const int64_t c = 8 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (c >= j.pitch) return;
    const int64_t step = gridDim.y;
    for (int64_t r = blockIdx.y; r < j.rows; r += kRowBatch * step) {
        PadLoad l[kRowBatch];
#pragma unroll
        for (int i = 0; i < kRowBatch; ++i)
            if (r + i * step < j.rows) l[i] = pad_load(j, r + i * step, c);
#pragma unroll
        for (int i = 0; i < kRowBatch; ++i)
            if (r + i * step < j.rows) pad_store(j, r + i * step, c, l[i]);
    }
}

// The same copy with bulk copies, for rows that fit a shared-memory stage:
// a chunk of whole source rows is fetched as the 16-byte granules that hold
// it (the granules contain bytes of the rows, so the fetch stays in the
// allocation's pages), realigned row by row into an output buffer whose
// rows have the destination pitch (slots past `cols` zero), and written
// back with one bulk store.  Same pipeline shape as widen_flat_kernel.
struct RowsJob {
    const uint16_t *src;
    int64_t rows, cols;
    uint16_t *dst;
    int64_t pitch;
    int64_t rows_per_chunk;  // whole rows per chunk, >= 1
};

constexpr int kRowsCap = 32768;  // bytes per input stage and per output buffer
constexpr int kRowsInStages = 4;
constexpr int kRowsOut = 3;
constexpr int kRowsThreads = 512;
constexpr int kRowsSmem = kRowsInStages * kRowsCap + kRowsOut * kRowsCap + 8 * kRowsInStages + 128;
static_assert(kRowsSmem <= 232448, "over the per-CTA shared-memory limit");
static_assert(kRowsOut >= 3, "an output buffer is rewritten two chunks after its store was confirmed read");

struct RowsChunk {
    uintptr_t load;     // 16-byte aligned start of the fetched granules
    uint32_t in_bytes;  // fetched bytes (a multiple of 16)
    uint32_t shift;     // byte offset of the chunk's first element in them
    int64_t rows;       // rows in the chunk
    uint16_t *dst;
    uint32_t out_bytes;
};

__device__ __forceinline__ RowsChunk rows_chunk(const RowsJob &j, int64_t k)
{
    RowsChunk c;
    const int64_t r0 = k * j.rows_per_chunk;
    const int64_t r1 = r0 + j.rows_per_chunk < j.rows ? r0 + j.rows_per_chunk : j.rows;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(j.src + r0 * j.cols);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(j.src + r1 * j.cols);
    c.load = a0 & ~static_cast<uintptr_t>(15);
    c.in_bytes = static_cast<uint32_t>(((a1 + 15) & ~static_cast<uintptr_t>(15)) - c.load);
    c.shift = static_cast<uint32_t>(a0 - c.load);
    c.rows = r1 - r0;
    c.dst = j.dst + r0 * j.pitch;
    c.out_bytes = static_cast<uint32_t>(c.rows * j.pitch * 2);
    return c;
}

__global__ void __launch_bounds__(kRowsThreads, 1)
    pad_rows_kernel(const RowsJob j0, const RowsJob j1, int *status, uint64_t timeout_ns)
{
    extern __shared__ __align__(128) uint8_t rsm[];
    const uint32_t base = (smem_u32(rsm) + 127u) & ~127u;
    const uint32_t in0 = base;
    const uint32_t out0 = base + kRowsInStages * kRowsCap;
    const uint32_t bar0 = out0 + kRowsOut * kRowsCap;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t c0 = (j0.rows + j0.rows_per_chunk - 1) / j0.rows_per_chunk;
    const int64_t total = c0 + (j1.rows > 0 ? (j1.rows + j1.rows_per_chunk - 1) / j1.rows_per_chunk : 0);
    const int64_t mine = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto job_of = [&](int64_t i, int64_t &k) -> const RowsJob & {
        const int64_t g = blockIdx.x + i * gridDim.x;
        k = g < c0 ? g : g - c0;
        return g < c0 ? j0 : j1;
    };
    auto issue = [&](int64_t i) {
        int64_t k;
        const RowsChunk c = rows_chunk(job_of(i, k), k);
        const int st = static_cast<int>(i % kRowsInStages);
        mbar_arrive_expect_tx(bar0 + 8 * st, c.in_bytes);
        bulk_load_g2s(in0 + st * kRowsCap, reinterpret_cast<const void *>(c.load), c.in_bytes, bar0 + 8 * st);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < kRowsInStages; ++st) mbar_init(bar0 + 8 * st, 1);
        fence_mbar_init();
        for (int64_t i = 0; i < mine && i < kRowsInStages; ++i) issue(i);
    }
    __syncthreads();
    int64_t issued = mine < kRowsInStages ? mine : kRowsInStages;
    int64_t i = 0;
    for (; i < mine; ++i) {
        const int st = static_cast<int>(i % kRowsInStages);
        const uint32_t parity = static_cast<uint32_t>((i / kRowsInStages) & 1);
        const uint32_t ob = out0 + static_cast<uint32_t>(i % kRowsOut) * kRowsCap;
        bool late = false;
        if (!mbar_try_wait(bar0 + 8 * st, parity)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar0 + 8 * st, parity))
                if (globaltimer_ns() - t0 > timeout_ns) {
                    late = true;
                    break;
                }
        }
        int64_t k;
        const RowsJob &j = job_of(i, k);
        const RowsChunk c = rows_chunk(j, k);
        if (!late) {
            // Output unit u = (row rr, 16-byte unit c8) holds 8 fp16 whose
            // source starts at byte shift + 2 * (rr * cols + 8 * c8) of the
            // stage.  Each thread walks units tid, tid + T, ... carrying
            // (rr, c8) forward instead of dividing per unit.
            const uint32_t ib = in0 + st * kRowsCap;
            const uint32_t per_row = static_cast<uint32_t>(j.pitch / 8);
            const uint32_t cols = static_cast<uint32_t>(j.cols);
            const uint32_t units = static_cast<uint32_t>(c.rows) * per_row;
            const uint32_t step_r = kRowsThreads / per_row, step_c = kRowsThreads - step_r * per_row;
            uint32_t rr = threadIdx.x / per_row, c8 = threadIdx.x - rr * per_row;
            for (uint32_t u = threadIdx.x; u < units; u += kRowsThreads) {
                const uint32_t b = c.shift + 2 * (rr * cols + 8 * c8);
                const uint32_t sh = b & 15u, ba = b & ~15u, col = 8 * c8;
                const uint4 lo = ld_shared_v4(ib + ba);
                const uint4 hi = sh ? ld_shared_v4(ib + ba + 16) : make_uint4(0, 0, 0, 0);
                uint32_t o[4];
                realign16(lo, hi, sh, o);
                if (col + 8 > cols) {
                    const int valid = col < cols ? static_cast<int>(cols - col) : 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t keep =
                            (2 * q < valid ? 0x0000FFFFu : 0u) | (2 * q + 1 < valid ? 0xFFFF0000u : 0u);
                        o[q] &= keep;
                    }
                }
                st_shared_v4(ob + 16 * u, o[0], o[1], o[2], o[3]);
                c8 += step_c;
                rr += step_r;
                if (c8 >= per_row) {
                    c8 -= per_row;
                    ++rr;
                }
            }
            fence_proxy_async_smem();
        }
        if (__syncthreads_or(late)) break;
        if (threadIdx.x == 0) {
            bulk_store_s2g(c.dst, ob, c.out_bytes);
            bulk_commit();
            if (issued < mine) {
                issue(issued);
                ++issued;
            }
            bulk_wait_read<kRowsOut - 2>();  // frees the buffer of chunk i + 2
        }
    }
    if (threadIdx.x == 0) {
        if (i < mine) {
            atomicCAS(status, 0, static_cast<int>(GEMMPIPE_ERR_TIMEOUT));
            for (int64_t q = i; q < issued; ++q) {
                const int st = static_cast<int>(q % kRowsInStages);
                const uint32_t parity = static_cast<uint32_t>((q / kRowsInStages) & 1);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar0 + 8 * st, parity))
                    if (globaltimer_ns() - t0 > timeout_ns) break;
            }
        }
        bulk_wait<0>();
    }
    __syncthreads();
}

__global__ void zero_fill_kernel(uint8_t *dst, int64_t bytes)
{
    pdl_wait();
    pdl_launch_dependents();
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
    pdl_wait();
    pdl_launch_dependents();
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

// Launches with programmatic dependent launch allowed: every kernel here
// starts with pdl_wait, so it may be scheduled while the previous grid on
// the stream finishes.
template <class... P, class... A>
cudaError_t launch_pdl(void (*k)(P...), dim3 grid, int threads, cudaStream_t s, A &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Blocks of `threads` threads of kernel k resident on one SM (cached per
// kernel; 8 if the query fails).
template <class K>
int resident_blocks(K k, int threads)
{
    static std::atomic<int> cached{0};
    int n = cached.load();
    if (n > 0) return n;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, 0) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 8;
    }
    cached.store(n);
    return n;
}

cudaError_t launch_widen_jobs(const WidenJob &ja, const WidenJob &jb, int sms, cudaStream_t s);

cudaError_t launch_widen_s8_f16(const int8_t *A, int64_t rowsA, int64_t colsA, uint16_t *A16, int64_t pitchA,
                                const int8_t *B, int64_t rowsB, int64_t colsB, uint16_t *B16, int64_t pitchB,
                                int sms, cudaStream_t s)
{
    const auto flat = [](const void *src, const void *dst, int64_t cols, int64_t pitch) {
        return cols % 16 == 0 && pitch == cols && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
               (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    };
    if (flat(A, A16, colsA, pitchA) && flat(B, B16, colsB, pitchB)) {
        static std::atomic<int> attr_done[128];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
        if (!attr_done[dev].load()) {
            e = cudaFuncSetAttribute(widen_flat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFlatSmem);
            if (e != cudaSuccess) return e;
            attr_done[dev].store(1);
        }
        int *st = nullptr;
        if ((e = status_word(&st)) != cudaSuccess) return e;
        const FlatJob fa{A, A16, rowsA * colsA};
        const FlatJob fb{B, B16, rowsB * colsB};
        const int64_t chunks = (fa.n + kFlatChunk - 1) / kFlatChunk + (fb.n + kFlatChunk - 1) / kFlatChunk;
        const int grid = static_cast<int>(chunks < sms ? chunks : sms);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid > 0 ? grid : 1, 1, 1);
        cfg.blockDim = dim3(kFlatThreads, 1, 1);
        cfg.dynamicSmemBytes = kFlatSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, widen_flat_kernel, fa, fb, st, static_cast<uint64_t>(2000000000ull));
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    return launch_widen_jobs(WidenJob{A, rowsA, colsA, colsA, A16, pitchA, pitchA},
                             WidenJob{B, rowsB, colsB, colsB, B16, pitchB, pitchB}, sms, s);
}

cudaError_t launch_widen_s8_f16_cols(const int8_t *src, int64_t rows, int64_t cols, int64_t spitch, uint16_t *dst,
                                     int64_t dpitch, int sms, cudaStream_t s)
{
    const WidenJob j{src, rows, cols, spitch, dst, dpitch, (cols + 7) / 8 * 8};
    return launch_widen_jobs(j, WidenJob{src, 0, cols, spitch, dst, dpitch, j.dcols}, sms, s);
}

cudaError_t launch_widen_jobs(const WidenJob &ja, const WidenJob &jb, int sms, cudaStream_t s)
{
    const int64_t rowsA = ja.rows, rowsB = jb.rows;
    const int threads = 128;
    const int64_t maxpitch = ja.dcols > jb.dcols ? ja.dcols : jb.dcols;
    const int64_t gx = ((maxpitch + 15) / 16 + threads - 1) / threads;
    const int64_t maxrows = rowsA > rowsB ? rowsA : rowsB;
    // One resident wave of blocks over both matrices, and at least a whole
    // batch of rows per thread.
    const int64_t wave = static_cast<int64_t>(sms) * resident_blocks(widen_s8_f16_kernel, threads);
    int64_t gy = (wave / 2 + gx - 1) / gx;
    if (gy * kRowBatch > maxrows) gy = (maxrows + kRowBatch - 1) / kRowBatch;
    gy = gy < 1 ? 1 : (gy > maxrows ? maxrows : gy);
    gy = gy > 65535 ? 65535 : gy;
    if (gx > 2147483647) return cudaErrorInvalidValue;
    return launch_pdl(widen_s8_f16_kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 2), threads, s,
                      ja, jb);
}

// Whole rows per bulk-copy chunk, 0 when a row does not fit a stage (the
// fetched granules of R rows span at most 2*R*cols + 30 bytes and the
// realigning reads look 16 bytes past the last output unit's source).
int64_t rows_per_chunk(int64_t cols, int64_t pitch, const uint16_t *dst)
{
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0 || pitch % 8 != 0) return 0;
    const int64_t w = 2 * (cols > pitch ? cols : pitch);
    return (kRowsCap - 64) / w;
}

cudaError_t launch_pad_f16(const uint16_t *src0, int64_t rows0, int64_t cols0, uint16_t *dst0, int64_t pitch0,
                           const uint16_t *src1, int64_t rows1, int64_t cols1, uint16_t *dst1, int64_t pitch1,
                           int sms, cudaStream_t s)
{
    // rows1 == 0: one job only.
    const int64_t r0 = rows_per_chunk(cols0, pitch0, dst0);
    const int64_t r1 = rows1 > 0 ? rows_per_chunk(cols1, pitch1, dst1) : 1;
    if (r0 > 0 && r1 > 0 && rows0 > 0) {
        static std::atomic<int> attr_done[128];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
        if (!attr_done[dev].load()) {
            e = cudaFuncSetAttribute(pad_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsSmem);
            if (e != cudaSuccess) return e;
            attr_done[dev].store(1);
        }
        int *st = nullptr;
        if ((e = status_word(&st)) != cudaSuccess) return e;
        const RowsJob a{src0, rows0, cols0, dst0, pitch0, r0};
        const RowsJob b{src1, rows1, cols1, dst1, pitch1, r1};
        const int64_t chunks = (rows0 + r0 - 1) / r0 + (rows1 > 0 ? (rows1 + r1 - 1) / r1 : 0);
        const int grid = static_cast<int>(chunks < sms ? chunks : sms);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid > 0 ? grid : 1, 1, 1);
        cfg.blockDim = dim3(kRowsThreads, 1, 1);
        cfg.dynamicSmemBytes = kRowsSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, pad_rows_kernel, a, b, st, static_cast<uint64_t>(2000000000ull));
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const PadJob j0{src0, rows0, cols0, dst0, pitch0};
    const PadJob j1{src1, rows1, cols1, dst1, pitch1};
    const int threads = 128;
    const int64_t maxpitch = pitch0 > pitch1 ? pitch0 : pitch1;
    const int64_t maxrows = rows0 > rows1 ? rows0 : rows1;
    const int64_t gx = (maxpitch / 8 + threads - 1) / threads;
    const unsigned gz = rows1 > 0 ? 2u : 1u;
    const int64_t wave = static_cast<int64_t>(sms) * resident_blocks(pad_f16_kernel, threads);
    int64_t gy = (wave / gz + gx - 1) / gx;
    if (gy * kRowBatch > maxrows) gy = (maxrows + kRowBatch - 1) / kRowBatch;
    gy = gy < 1 ? 1 : (gy > maxrows ? maxrows : gy);
    gy = gy > 65535 ? 65535 : gy;
    if (gx > 2147483647) return cudaErrorInvalidValue;
    return launch_pdl(pad_f16_kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), gz), threads, s, j0,
                      j1);
}

cudaError_t launch_zero_fill(void *dst, int64_t bytes, int sms, cudaStream_t s)
{
    const int64_t need = (bytes / 16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 4;
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    return launch_pdl(zero_fill_kernel, dim3(grid), 256, s, static_cast<uint8_t *>(dst), bytes);
}

cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, int sms, cudaStream_t s)
{
    const int64_t need = (bytes / 16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    return launch_pdl(copy_kernel, dim3(grid), 256, s, static_cast<uint8_t *>(dst), static_cast<const uint8_t *>(src),
                      bytes);
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
