// gemm_imma.cu -- the pages' own kernel design on sm_103a, kept as a
// comparison path for INT8: warp-level integer MMA (mma.sync m16n8k32,
// s8 x s8 -> s32) fed by a cp.async shared-memory ring.
//
// "Pipeline GPU Kernel", Steps 1-3: each CTA owns a 128 x 128 tile of C;
// the K loop is software-pipelined with an S-stage ring of cp.async copies
// (S = 2 is the page's double buffer, S = 4 the default), so the copies of
// k-block n + S - 1 are in flight while the tensor cores work on k-block n.
// The arithmetic is exact integer accumulation (int32, wrapping like the
// tcgen05 path).
//
// B is consumed transposed (N x K, K contiguous) so both operands feed
// ldmatrix with 16-byte k-rows; transpose_s8_kernel makes that copy (the
// blog page's shared-memory tiled transpose, with coalesced reads and
// writes).  Requirements: A and the transposed B 16-byte aligned, K a
// multiple of 16 (whole 16-byte row chunks); M, N arbitrary.
#include <cstdint>

#include "ptx.cuh"
#include "variants.h"

namespace gp {

namespace {

constexpr int kIBM = 128, kIBN = 128, kIBK = 64;  // tile; BK in int8 (bytes)
constexpr int kIThreads = 256;                  // 8 warps: 2 (m) x 4 (n), warp tile 64 x 32
constexpr int kIStageBytes = (kIBM + kIBN) * kIBK;  // 16 KiB
constexpr int kIDefaultStages = 4;

// A stage row holds 64 bytes = four 16-byte chunks; chunk c of row r is
// stored at chunk c ^ ((r >> 1) & 3), which makes every ldmatrix (eight
// rows, one chunk each) and every cp.async row write bank-conflict free.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c)
{
    return r * 64 + ((c ^ ((r >> 1) & 3u)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct ImmaParams {
    const int8_t *A;   // M x K, row pitch K
    const int8_t *BT;  // N x K, row pitch ldbt
    int32_t *C;        // M x N, row pitch N
    int64_t M, N, K, ldbt;
};

// Copies k-block kb of this CTA's A rows and BT rows into stage `st`:
// 2 x 128 rows x 4 chunks = 1024 chunks, four per thread.  Chunks outside
// the matrices are zero-filled (source size 0, a valid dummy address).
__device__ __forceinline__ void load_stage(const ImmaParams &p, uint32_t sbase, int st, int64_t kb, int64_t m0,
                                           int64_t n0)
{
    const uint32_t sa = sbase + st * kIStageBytes;
    const uint32_t sb = sa + kIBM * kIBK;
    const int64_t k0 = kb * kIBK;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * kIThreads;  // 0..1023
        const int half = idx >> 9;                    // 0: A, 1: BT
        const int r = (idx >> 2) & 127, c = idx & 3;
        const int64_t k = k0 + 16 * c;
        if (half == 0) {
            const int64_t row = m0 + r;
            const bool ok = row < p.M && k < p.K;
            cp_async16(sa + swz(r, c), ok ? p.A + row * p.K + k : p.A, ok ? 16u : 0u);
        } else {
            const int64_t row = n0 + r;
            const bool ok = row < p.N && k < p.K;
            cp_async16(sb + swz(r, c), ok ? p.BT + row * p.ldbt + k : p.BT, ok ? 16u : 0u);
        }
    }
}

template <int kIStages>
__global__ void __launch_bounds__(kIThreads, 2) gemm_imma_kernel(const ImmaParams p)
{
    static_assert(kIStages >= 2, "the ring keeps kIStages - 1 k-blocks in flight");
    extern __shared__ __align__(128) uint8_t ism[];
    const uint32_t sbase = (smem_u32(ism) + 127u) & ~127u;
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = warp >> 2, wn = warp & 3;  // warp tile at rows 64 wm, columns 32 wn
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kIBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kIBN;
    const int64_t nkb = (p.K + kIBK - 1) / kIBK;

    int acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;

    // Prologue: the first S - 1 k-blocks in flight (one group each, empty
    // groups past the end keep the count uniform).
#pragma unroll
    for (int st = 0; st < kIStages - 1; ++st) {
        if (st < nkb) load_stage(p, sbase, st, st, m0, n0);
        cp_async_commit();
    }
    // ldmatrix lane addressing: lanes 0-7 / 8-15 / 16-23 / 24-31 give the
    // row addresses of the four 8 x 8 (b16) matrices.
    const int lrow = lane & 7, lsel = lane >> 3;
    for (int64_t kb = 0; kb < nkb; ++kb) {
        cp_async_wait<kIStages - 2>();  // k-block kb has landed (this thread's copies)
        __syncthreads();                // ... and everyone's; stage (kb - 1) % S is free
        const int64_t nxt = kb + kIStages - 1;
        if (nxt < nkb) load_stage(p, sbase, static_cast<int>(nxt % kIStages), nxt, m0, n0);
        cp_async_commit();
        const uint32_t sa = sbase + static_cast<int>(kb % kIStages) * kIStageBytes;
        const uint32_t sb = sa + kIBM * kIBK;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {  // two k32 steps per 64-byte k-block
            uint32_t af[4][4], bf[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // A 16 x 32 bytes: matrices (rows 0-7 | 8-15) x (bytes 0-15 | 16-31).
                const uint32_t r = 64 * wm + 16 * i + lrow + 8 * (lsel & 1);
                const uint32_t c = 2 * ks + (lsel >> 1);
                ldmatrix_x4(sa + swz(r, c), af[i][0], af[i][1], af[i][2], af[i][3]);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // BT 16 columns x 32 bytes: (cols 0-7, bytes 0-15), (0-7, 16-31),
                // (8-15, 0-15), (8-15, 16-31) -> b0, b1 of two n8 tiles.
                const uint32_t r = 32 * wn + 16 * j + lrow + 8 * (lsel >> 1);
                const uint32_t c = 2 * ks + (lsel & 1);
                ldmatrix_x4(sb + swz(r, c), bf[2 * j][0], bf[2 * j][1], bf[2 * j + 1][0], bf[2 * j + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
    }
    cp_async_wait<0>();

    // Accumulator (i, j): rows 64 wm + 16 i + g (+ 8), columns 32 wn + 8 j +
    // 2 t (+ 1), g = lane / 4, t = lane % 4.
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = m0 + 64 * wm + 16 * i + g + 8 * h;
            if (row >= p.M) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t col = n0 + 32 * wn + 8 * j + 2 * t;
                int32_t *dst = p.C + row * p.N + col;
                const int v0 = acc[i][j][2 * h], v1 = acc[i][j][2 * h + 1];
                if (col + 1 < p.N && ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0)) {
                    *reinterpret_cast<int2 *>(dst) = make_int2(v0, v1);
                } else {
                    if (col < p.N) dst[0] = v0;
                    if (col + 1 < p.N) dst[1] = v1;
                }
            }
        }
}

// B (K x N, N contiguous) -> BT (N x K, row pitch ldbt, K contiguous) through
// a 64 x 64 shared-memory tile: 16-byte row reads, 16-byte row writes.
__global__ void __launch_bounds__(256) transpose_s8_kernel(const int8_t *B, int64_t K, int64_t N, int8_t *BT,
                                                           int64_t ldbt)
{
    __shared__ uint8_t tile[64][64 + 4];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t k0 = static_cast<int64_t>(blockIdx.y) * 64, n0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 16;  // 64 rows x 4 pieces of 16 bytes
    {
        const int64_t k = k0 + r;
        const int8_t *src = B + k * N + n0 + c;
        if (k < K && n0 + c + 16 <= N && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            const uint4 v = *reinterpret_cast<const uint4 *>(src);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int b = 0; b < 16; ++b) tile[r][c + b] = static_cast<uint8_t>((w[b / 4] >> (8 * (b % 4))) & 0xFFu);
        } else {
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const int64_t n = n0 + c + b;
                tile[r][c + b] = (k < K && n < N) ? static_cast<uint8_t>(B[k * N + n]) : 0u;
            }
        }
    }
    __syncthreads();
    const int64_t n = n0 + r;
    if (n >= N) return;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t x = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) x |= static_cast<uint32_t>(tile[c + 4 * q + b][r]) << (8 * b);
        w[q] = x;
    }
    const int64_t k = k0 + c;
    if (k + 16 <= ldbt) {
        *reinterpret_cast<uint4 *>(BT + n * ldbt + k) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        for (int b = 0; b < 16 && k + b < ldbt; ++b) BT[n * ldbt + k + b] = static_cast<int8_t>((w[b / 4] >> (8 * (b % 4))) & 0xFFu);
    }
}

}  // namespace

bool imma_supported(const int8_t *A, int64_t K)
{
    return K % 16 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
}

int64_t imma_bt_pitch(int64_t K) { return (K + 15) / 16 * 16; }

cudaError_t launch_transpose_s8(const int8_t *B, int64_t K, int64_t N, int8_t *BT, int64_t ldbt, cudaStream_t s)
{
    const int64_t gx = (N + 63) / 64, gy = (K + 63) / 64;
    if (gx > 2147483647 || gy > 65535) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, transpose_s8_kernel, B, K, N, BT, ldbt);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int S>
cudaError_t launch_imma_stages(const ImmaParams &p, dim3 grid, cudaStream_t s)
{
    constexpr int smem = S * kIStageBytes + 128;
    static bool attr_done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(gemm_imma_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kIThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_imma_kernel<S>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int imma_stages(int requested) { return requested == 2 ? 2 : kIDefaultStages; }

cudaError_t launch_imma_s8(const int8_t *A, const int8_t *BT, int64_t ldbt, int32_t *C, int64_t M, int64_t N,
                           int64_t K, int stages, cudaStream_t s)
{
    const int64_t gx = (N + kIBN - 1) / kIBN, gy = (M + kIBM - 1) / kIBM;
    if (gx > 2147483647 || gy > 65535) return cudaErrorInvalidValue;
    const ImmaParams p{A, BT, C, M, N, K, ldbt};
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
    return imma_stages(stages) == 2 ? launch_imma_stages<2>(p, grid, s) : launch_imma_stages<4>(p, grid, s);
}

void imma_plan_info(VariantInfo *f, int stages)
{
    const int S = imma_stages(stages);
    *f = VariantInfo{2, 1, 0, kIBM, kIBN, kIBK, S, 0, 0, kIThreads, S * kIStageBytes + 128, 0};
}

}  // namespace gp
