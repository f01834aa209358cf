// gemmpipe_api.cpp -- the C ABI declared in include/gemmpipe.h: argument
// checks, plan selection, tensor-map encoding, the INT8 workspace, kernel
// timing and the device status word.
#include "gemmpipe.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "variants.h"

namespace {

using gp::GemmParams;
using gp::Variant;

constexpr int64_t kMaxDim = 2147483647;  // 2^31 - 1
constexpr int kBM = 128, kBK = 64;
constexpr int64_t kInt8ChunkK = 1024;  // k values per exact fp32 partial (1024 * 2^14 = 2^24)

std::mutex g_mu;
std::atomic<int64_t> g_launches{0};

// ------------------------------------------------------------- device info

struct DeviceInfo {
    int ok = 0;
    int major = 0, minor = 0;
    int sms = 0;
    int smem_optin = 0;
};

gemmpipe_status_t device_info(DeviceInfo *out, int *dev_out)
{
    static DeviceInfo cache[128];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
        cudaGetLastError();
        return GEMMPIPE_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = cache[dev];
    if (!d.ok) {
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMMPIPE_ERR_UNSUPPORTED_DEVICE;
        }
        d.ok = 1;
    }
    if (d.major != 10 || d.minor != 3) return GEMMPIPE_ERR_UNSUPPORTED_DEVICE;
    *out = d;
    if (dev_out) *dev_out = dev;
    return GEMMPIPE_OK;
}

// -------------------------------------------------------- argument checks

gemmpipe_status_t check_pointer(const void *p, int align)
{
    if (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(align)) return GEMMPIPE_ERR_INVALID_VALUE;
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof(a));
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_INVALID_VALUE;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return GEMMPIPE_ERR_INVALID_VALUE;
    return GEMMPIPE_OK;
}

// Checks that need no GPU (sizes, null pointers, element alignment).
gemmpipe_status_t check_shape(int64_t M, int64_t N, int64_t K, const void *A, const void *B, const void *C,
                              int ab_bytes, int c_bytes)
{
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMMPIPE_ERR_INVALID_VALUE;
    // No matrix (or padded copy of one) may hold 2^56 elements or more, so
    // that byte counts of operands and workspaces stay far inside int64.
    constexpr int64_t kMaxElems = int64_t(1) << 56;
    if ((K > 0 && M > kMaxElems / (K + 8)) || (N > 0 && K > kMaxElems / (N + 8)) ||
        (N > 0 && M > kMaxElems / N))
        return GEMMPIPE_ERR_INVALID_VALUE;
    // The kernels number C's tiles in 32 bits.  Counted in the smallest
    // tile (128 x 128), a C of 2^31 tiles holds 2^45 values: no device holds
    // it, so such sizes are refused before anything is launched.
    if (((M + 127) / 128) * ((N + 127) / 128) > INT32_MAX) return GEMMPIPE_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMMPIPE_OK;
    if (!C) return GEMMPIPE_ERR_INVALID_VALUE;
    if (K > 0 && (!A || !B)) return GEMMPIPE_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(C) % c_bytes) return GEMMPIPE_ERR_INVALID_VALUE;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) % ab_bytes) || (reinterpret_cast<uintptr_t>(B) % ab_bytes)))
        return GEMMPIPE_ERR_INVALID_VALUE;
    return GEMMPIPE_OK;
}

gemmpipe_status_t check_device_pointers(int64_t K, const void *A, const void *B, const void *C, int ab_bytes,
                                        int c_bytes)
{
    gemmpipe_status_t s = check_pointer(C, c_bytes);
    if (s != GEMMPIPE_OK) return s;
    if (K > 0) {
        if ((s = check_pointer(A, ab_bytes)) != GEMMPIPE_OK) return s;
        if ((s = check_pointer(B, ab_bytes)) != GEMMPIPE_OK) return s;
    }
    return GEMMPIPE_OK;
}

// ------------------------------------------------------------------ plans

struct Override {
    int producer = -1, bn = 0, stages = 0, pair = -1, split = -1;
    int bk = 0;  // k values per stage: 0 automatic (64), or 64 / 128
};
Override g_override;

struct StallHook {
    int64_t kb = -1;
    int timeout_ms = 0;
};
StallHook g_stall;

struct TraceHook {
    unsigned long long *buf = nullptr;
    int64_t n = 0;
};
TraceHook g_trace_hook;

struct Plan {
    const Variant *v = nullptr;
    int grid = 0;
    int64_t tiles = 0, m_tiles = 0, num_kb = 0, kb_per_chunk = 0, group_m = 1;
    int64_t units = 0, dp_tiles = 0, sk_tiles = 0;
    int64_t slots = 0;  // co-resident units (CTAs or CTA pairs)
    int vec_store = 0;
    // CTAs per unit: 1, a CTA pair (2), or a quad of two pairs (4).
    int cluster() const { return v->info.pair == 2 ? 4 : (v->info.pair ? 2 : 1); }
    int64_t split_ctas() const { return cluster() * units; }
    int64_t split_bytes() const;  // stream-K partials + flags (0: none)
    void run_whole_tiles()
    {
        units = tiles < slots ? tiles : slots;
        dp_tiles = tiles;
        sk_tiles = 0;
        grid = static_cast<int>(cluster() * units);
    }
};

// Stream-K flags: one per epilogue warp of each CTA, in a fixed region at
// the start of the split workspace that holds nothing but epochs (partial
// sums of a plan with a larger grid never land where a flag of another plan
// is read), so a flag equals the current epoch only once this launch has
// published it.  Launches beyond kMaxSplitCtas CTAs run whole tiles.
constexpr int64_t kSplitFlagsPerCta = 8;
constexpr int64_t kMaxSplitCtas = 2048;
constexpr int64_t kSplitFlagBytes = kMaxSplitCtas * kSplitFlagsPerCta * 4;

// Fewest k-blocks a stream-K unit is given when tiles alone cannot fill the
// grid: below this the ring's fill and the fix-up cost more than the idle
// SMs they replace.
constexpr int64_t kMinSplitKb = 8;
// Fewest k values a split must take off each single-CTA unit to pay for
// its fix-up when there are fewer tiles than units.
constexpr int64_t kMinSavedK = 1536;

// Dense fp16 tensor flops per byte of HBM traffic at which GB300 turns from
// memory- to compute-bound (about 2.2 PFLOP/s over 7.9 TB/s; a copy and a
// cuBLAS GEMM measure 1.9 PFLOP/s over 6.8 TB/s, the same ratio).
constexpr double kMachineBalance = 280.0;

int64_t Plan::split_bytes() const
{
    if (sk_tiles == 0) return 0;
    return kSplitFlagBytes + split_ctas() * static_cast<int64_t>(v->info.BM) * v->info.BN * 4;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

const Variant *find_variant(int int_out, int convert, int producer, int bn, int stages, int pair, int bk = 64)
{
    const Variant *tab = nullptr;
    const int n = int_out ? gp::variants_s8(&tab) : gp::variants_f16(&tab);
    for (int i = 0; i < n; ++i) {
        const gp::VariantInfo &f = tab[i].info;
        if (f.producer == producer && f.convert == convert && f.BN == bn && f.pair == pair && !f.traced &&
            f.BK == bk && (stages == 0 || f.stages == stages))
            return &tab[i];
    }
    return nullptr;
}

// The trace-stamping copy of a variant, if one was compiled.
const Variant *traced_twin(const Variant *v)
{
    const Variant *tab = nullptr;
    const int n = v->info.int_out ? gp::variants_s8(&tab) : gp::variants_f16(&tab);
    for (int i = 0; i < n; ++i) {
        const gp::VariantInfo &f = tab[i].info;
        if (f.traced && f.producer == v->info.producer && f.convert == v->info.convert && f.BN == v->info.BN &&
            f.pair == v->info.pair && f.stages == v->info.stages && f.int_out == v->info.int_out &&
            f.BK == v->info.BK)
            return &tab[i];
    }
    return nullptr;
}

// INT8 operands the converter variant can take straight from the caller:
// TMA needs 16-byte aligned bases and row pitches (K and N multiples of 16
// int8).  It is taken only when asked for (producer override 0): widening
// inside the kernel redoes the conversion of every operand tile for every
// output tile that reads it through the load/store pipe while the tensor
// cores read shared memory, and in a CTA pair each k-block needs a
// cross-CTA release-arrive from the peer's converters; measured, both make
// it slower than one widening pass plus the fp16 kernel.
bool s8_convert_ok(const void *A, int64_t K, const void *B, int64_t N)
{
    if (!(aligned16(A) && aligned16(B) && K % 16 == 0 && N % 16 == 0)) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_override.producer == 0;
}

// The legacy warp-MMA INT8 path (producer override 2): A read in place,
// B transposed into the workspace.
bool imma_wanted(const int8_t *A, int64_t K)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_override.producer != 2) return false;
    }
    return gp::imma_supported(A, K);
}

int64_t imma_workspace_bytes(int64_t N, int64_t K) { return N * gp::imma_bt_pitch(K); }

// The plan of one GEMM.  fp16 operands (or INT8 calls' widened copies) when
// convert is false; int8 operands read by TMA and widened in the kernel when
// convert is true.
gemmpipe_status_t make_plan(bool int_out, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                            const void *B, int64_t ldb, const void *C, int64_t ldc, const DeviceInfo &d, Plan *pl,
                            bool convert = false, bool split_ok = true)
{
    Override ov;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ov = g_override;
    }
    const int esz = convert ? 1 : 2;
    const bool tma_ok = aligned16(A) && aligned16(B) && (lda * esz) % 16 == 0 && (ldb * esz) % 16 == 0;
    int producer = tma_ok ? 0 : 1;
    if (ov.producer == 1) producer = 1;
    if (int_out) producer = 0;  // widened operands are always TMA-describable
    int bn = N <= 128 ? 128 : 256;
    // Small problems: when the 256 x 256 pair tiles would number at most a
    // quarter of the SM pairs, single CTAs on 128 x 128 tiles spread the
    // same k-loop over four times as many SMs with a quarter of the
    // epilogue each (measured on GB300, L2 flushed, per step: INT8 512^3
    // 14.6 vs 17.4 us, FP16 512^3 11.5 vs 14.4, FP16 1024^3 14.3 vs 16.6,
    // INT8 1024^3 17.2 vs 18.4).
    const int64_t pair_tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + 255) / 256);
    const bool small = bn == 256 && 4 * pair_tiles <= d.sms / 2;
    if (small && ov.pair < 1) bn = 128;
    if (ov.bn) bn = ov.bn;
    // A CTA pair (256 x 256 or 256 x 512 tiles, cta_group::2 MMA) when both
    // dimensions exceed one 128-row / 128-column tile and TMA reads the
    // operands.  512-wide tiles exist for fp16 output only; elsewhere they
    // become 256-wide.
    const Variant *v = nullptr;
    // Quads (two pairs of 256 x 256 tiles sharing A): asked for (cta_pair
    // override 2), or by default when C's rows are off 16-byte boundaries.
    // Such a C is written with 4-byte stores, and there quads measured 3.5-9%
    // faster (FP16 4093x3001x4107 81.8 vs 86.2 us, 4096x3001x4096 79.8 vs
    // 82.9, 2000x3001x2000 41.0 vs 44.9, 8191x6001x4096 269.9 vs 274.8; INT8
    // 4093x3001x4107 87.9 vs 88.8), while on aligned C they gained or lost a
    // few percent by shape.
    const bool c_aligned = aligned16(C) && (ldc * 4) % 16 == 0;
    const bool want_quad = ov.pair == 2 || (ov.pair == -1 && !c_aligned && !convert);
    if (producer == 0 && bn >= 256 && M > kBM && N > 128 && ov.pair != 0) {
        if (want_quad && bn == 256) v = find_variant(int_out, convert ? 1 : 0, 0, 256, ov.stages, 2);
        // CTA pairs take six stages of 64 k; 128 k per stage (three stages)
        // only when asked for.  With the MMA issue on the whole warp, 64-k
        // stages measured faster (A/B in one process, kernel time: FP16
        // 4096^3 84.9 vs 87.9 us, INT8 4096^3 83.1 vs 84.8, FP16 8192^3 596
        // vs 604, 2048 x 4096^2 50.0 vs 52.5, 6144^3 258.2 vs 263.3).
        const bool bk128 = ov.bk == 128;
        if (!v && bk128) v = find_variant(int_out, convert ? 1 : 0, 0, bn, ov.stages, 1, 128);
        if (!v) v = find_variant(int_out, convert ? 1 : 0, 0, bn, ov.stages, 1);
        if (!v && bn == 512) v = find_variant(int_out, convert ? 1 : 0, 0, 256, ov.stages, 1);
        if (v && v->max_pairs() < 1) v = nullptr;
    }
    if (bn == 512 && (!v || !v->info.pair)) bn = 256;
    // Single CTAs take 128 k per stage when asked for (plan override), and
    // by default for fp16 with N <= 128 (the skinny, memory-bound case: each
    // A row is read 256 bytes at a time; A/B in one process, kernel time:
    // 16384 x 128 x 16384 112.1 vs 113.7 us, 16384 x 64 x 16384 111.5 vs
    // 112.6, 8192 x 128 x 8192 and 32768 x 128 x 8192 within 0.3%).
    const bool single_bk128 = ov.bk == 128 || (ov.bk == 0 && ov.stages == 0 && !int_out && N <= 128);
    if (!v && single_bk128 && producer == 0 && !convert) v = find_variant(int_out, 0, 0, bn, ov.stages, 0, 128);
    if (!v) v = find_variant(int_out, convert ? 1 : 0, producer, bn, ov.stages, 0);
    if (!v) v = find_variant(int_out, convert ? 1 : 0, producer, bn, 0, 0);
    if (!v) return GEMMPIPE_ERR_INTERNAL;
    if (v->info.smem_bytes > d.smem_optin) return GEMMPIPE_ERR_UNSUPPORTED_DEVICE;
    pl->v = v;
    bn = v->info.BN;
    const int64_t tile_m = v->info.pair ? 2 * kBM : kBM;
    const int64_t tile_n = v->info.pair == 2 ? 2 * bn : bn;
    pl->m_tiles = (M + tile_m - 1) / tile_m;
    pl->tiles = pl->m_tiles * ((N + tile_n - 1) / tile_n);
    // Already refused by the shape check (tile indices are 32-bit).
    if (pl->tiles > INT32_MAX) return GEMMPIPE_ERR_INVALID_VALUE;
    const int bk = v->info.BK;
    pl->num_kb = (K + bk - 1) / bk;
    pl->kb_per_chunk = int_out ? kInt8ChunkK / bk : pl->num_kb;
    // Persistent grid: at most one CTA (or CTA pair) per SM (pair) slot.
    // Whole tiles go round-robin; when they leave a partial last wave that
    // is at most 4/5 full, that wave and the one before it are spread over
    // all units as equal ranges of k-blocks (stream-K), so every unit does
    // the same work.  With fewer tiles than slots, all tiles are split over
    // as many units as keep at least kMinSplitKb k-blocks each, when that
    // cuts a unit's k-blocks to a third or less -- or, on single CTAs of a
    // compute-bound GEMM, by kMinSavedK k values or more.  Measured on
    // GB300: a split costs its fix-up and, with every SM streaming operands
    // at once, a slower k-loop (about 7 us on single CTAs), so it pays only
    // when the work per unit drops a lot.  Single CTAs, M = N = 1024 (64
    // tiles on 152 units), call time whole vs split: K = 2048 16.7 vs 18.7
    // us (1152 k fewer per unit), 3072 20.8 vs 19.3 (1728), 4096 23.4 vs
    // 21.0, 8192 38.9 vs 27.2; INT8 K = 2048 20.8 vs 21.4, 4096 29.5 vs
    // 27.1.  CTA pairs with 32 to 64 tiles on 76 pairs (N = K = 4096) stay
    // faster whole.
    // Quads (the plan for C rows off 16-byte boundaries, whose row-piece
    // stores make every item's epilogue long) split only a last wave at
    // most half full after two or more full waves (measured: 96 tiles on 36
    // quads 82.3 vs 79.6 us split vs whole, 48 tiles 40.9 vs 39.7, 384
    // tiles 271 vs 267; 120 tiles 92.9 vs 99.1).
    const int64_t slots = v->info.pair ? v->max_pairs() : d.sms;
    const int64_t T = pl->tiles;
    const bool split = split_ok && v->info.split_ok && ov.split != 0;
    pl->slots = slots;
    pl->run_whole_tiles();
    // A memory-bound GEMM (flops per compulsory byte below the machine
    // balance) whose tiles already occupy half the SMs or more gains
    // nothing from more SMs, only the fix-up traffic: its tiles stay whole.
    const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
    const double esz_in = convert ? 1.0 : 2.0;  // operand bytes the kernel reads
    const double bytes =
        esz_in * (static_cast<double>(M) * K + static_cast<double>(K) * N) + 4.0 * static_cast<double>(M) * N;
    const bool memory_bound = flops < kMachineBalance * bytes;
    if (split && T < slots) {
        const int64_t want = (T * pl->num_kb + kMinSplitKb - 1) / kMinSplitKb;
        const int64_t u = want < slots ? want : slots;
        // k values a unit computes fewer than with whole tiles.
        const int64_t saved_k = u > T ? (pl->num_kb - (T * pl->num_kb + u - 1) / u) * bk : 0;
        const bool pays = u >= 3 * T || (v->info.pair == 0 && !memory_bound && saved_k >= kMinSavedK);
        if (u > T && (ov.split == 1 || (pays && !(memory_bound && 2 * T >= slots)))) {
            pl->units = u;
            pl->dp_tiles = 0;
            pl->sk_tiles = T;
        }
    } else if (split && T > slots && T % slots != 0 && pl->num_kb > 1 &&
               (ov.split == 1 || (v->info.pair == 2 ? (2 * (T % slots) <= slots && T >= 2 * slots)
                                                    : 5 * (T % slots) <= 4 * slots))) {
        pl->sk_tiles = slots + T % slots;
        pl->dp_tiles = T - pl->sk_tiles;
    }
    pl->grid = static_cast<int>(pl->cluster() * pl->units);
    // Tile rows per group ~ sqrt(units): the tiles of a wave then cover
    // about sqrt(units) panels of A and as many of B, the fewest bytes.
    int64_t gm = 1;
    while ((gm + 1) * (gm + 1) <= pl->units) ++gm;
    pl->group_m = gm < pl->m_tiles ? gm : pl->m_tiles;
    pl->vec_store = aligned16(C) && (ldc * 4) % 16 == 0;
    return GEMMPIPE_OK;
}

// ------------------------------------------------------------ tensor maps

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static std::atomic<EncodeFn> fn{nullptr};
    EncodeFn f = fn.load();
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<EncodeFn>(p);
        fn.store(f);
    }
    return f;
}

// 2-D row-major tensor (rows x cols, pitch `ld` elements), zero fill
// outside it.  fp16: 128-byte swizzle, box 64 columns x box_rows rows.
// int8: no swizzle, box box_cols x box_rows.
bool encode_2d_any(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                   int box_rows, bool int8, bool swizzle128 = false)
{
    EncodeFn f = encode_fn();
    if (!f) return false;
    const int esz = int8 ? 1 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * esz)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             (int8 && !swizzle128) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows)
{
    return encode_2d_any(m, base, rows, cols, ld, 64, box_rows, false);
}

// B (rows x cols fp16, pitch ld, cols a multiple of 64) as 64 columns x
// rows x cols / 64 column groups, 128-byte swizzle; a box of box_rows rows
// and `groups` column groups lands as `groups` 64-column atoms, 8 KiB apart
// for 64-row boxes -- the layout of that many 2-D boxes.
bool encode_b_groups(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                     int groups)
{
    EncodeFn f = encode_fn();
    if (!f || cols % 64 != 0) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(groups)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C (rows x cols of 4-byte elements, pitch ld) for the epilogue's TMA
// stores: 32 x 32 boxes in the 128-byte swizzle of its staging tiles.
bool encode_c(CUtensorMap *m, void *C, int64_t rows, int64_t cols, int64_t ld, bool int_out)
{
    EncodeFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 4)};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, int_out ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ timing

struct Timing {
    bool enabled = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> gemm, aux;
    std::vector<cudaEvent_t> pool;
};
Timing g_timing;

cudaEvent_t take_event()
{
    if (!g_timing.pool.empty()) {
        cudaEvent_t e = g_timing.pool.back();
        g_timing.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}

struct TimedRegion {
    bool on = false;
    bool is_gemm;
    cudaStream_t s;
    cudaEvent_t a = nullptr, b = nullptr;
    TimedRegion(bool gemm, cudaStream_t st) : is_gemm(gemm), s(st)
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_timing.enabled) return;
        a = take_event();
        b = take_event();
        if (a && b && cudaEventRecord(a, s) == cudaSuccess) on = true;
    }
    void end()
    {
        if (!on) return;
        std::lock_guard<std::mutex> lk(g_mu);
        if (cudaEventRecord(b, s) == cudaSuccess) (is_gemm ? g_timing.gemm : g_timing.aux).push_back({a, b});
        on = false;
    }
};

// -------------------------------------------------------------- workspace

struct Workspace {
    void *ptr = nullptr;
    int64_t bytes = 0;
};
// Kinds of workspace per (device, stream).
enum WsKind { kWsOperands = 0, kWsSplit = 1, kWsHost = 2 };
std::map<std::tuple<int, cudaStream_t, int>, Workspace> g_ws;

// The (device, stream) workspace of one kind, at least `bytes` long.  A new
// stream-K workspace has its flags (the first zero_bytes bytes) zeroed on
// the stream before first use.
gemmpipe_status_t workspace(int dev, cudaStream_t s, int64_t bytes, void **out, int kind = kWsOperands,
                            int64_t zero_bytes = 0)
{
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[std::make_tuple(dev, s, kind)];
    if (w.bytes < bytes) {
        if (w.ptr) {
            cudaFree(w.ptr);  // synchronizes: earlier users of the buffer have finished
            w.ptr = nullptr;
            w.bytes = 0;
        }
        if (cudaMalloc(&w.ptr, static_cast<size_t>(bytes)) != cudaSuccess) {
            cudaGetLastError();
            w.ptr = nullptr;
            return GEMMPIPE_ERR_OUT_OF_MEMORY;
        }
        w.bytes = bytes;
        if (zero_bytes > 0 && cudaMemsetAsync(w.ptr, 0, static_cast<size_t>(zero_bytes), s) !=
                cudaSuccess) {
            cudaGetLastError();
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
            return GEMMPIPE_ERR_LAUNCH;
        }
    }
    *out = w.ptr;
    return GEMMPIPE_OK;
}

// ------------------------------------------------------------------- runs

std::atomic<uint32_t> g_epoch{0};

// Fills the stream-K fields of p: the split tiles' partial sums and flags in
// the stream's split workspace, and a fresh epoch.  Without that workspace
// the plan falls back to whole tiles.
void set_schedule(Plan &pl, int dev, cudaStream_t s, GemmParams &p)
{
    p.partials = nullptr;
    p.flags = nullptr;
    p.epoch = 0;
    if (pl.sk_tiles > 0) {
        void *ws = nullptr;
        if (pl.split_ctas() <= kMaxSplitCtas &&
            workspace(dev, s, pl.split_bytes(), &ws, kWsSplit, kSplitFlagBytes) == GEMMPIPE_OK) {
            p.flags = static_cast<uint32_t *>(ws);
            p.partials = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kSplitFlagBytes);
            uint32_t e = g_epoch.fetch_add(1) + 1;
            if (e == 0) e = g_epoch.fetch_add(1) + 1;  // 0 is the zeroed flags' value
            p.epoch = e;
        } else {
            pl.run_whole_tiles();
        }
    }
    p.m_tiles = pl.m_tiles;
    p.tiles = pl.tiles;
    p.group_m = pl.group_m;
    p.units = pl.units;
    p.dp_tiles = pl.dp_tiles;
    p.sk_work = pl.sk_tiles * pl.num_kb;
    p.num_kb = pl.num_kb;
    p.kb_per_chunk = pl.kb_per_chunk;
    p.vec_store = pl.vec_store;
}

gemmpipe_status_t run_plan(Plan pl, int dev, int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                           const uint16_t *B, int64_t ldb, void *C, int64_t ldc, cudaStream_t s)
{
    int b_groups = 0;
    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (pl.v->info.convert) {
        // int8: A box 64 (k) x 128 rows unswizzled; B in 128 x 64 atoms with
        // the 128-byte swizzle.
        if (!encode_2d_any(&ta, A, M, K, lda, kBK, kBM, true) ||
            !encode_2d_any(&tb, B, K, N, ldb, 128, kBK, true, true))
            return GEMMPIPE_ERR_INTERNAL;
    } else if (pl.v->info.producer == 0) {
        // Boxes: A 64 (k) x 128 rows, B 64 (n) x 64 (k); a pair CTA loads the
        // same boxes for its half -- or, when N is a multiple of 64, each
        // MMA's share of B in one 3-D box of 64-column groups.
        // A quad's CTA loads half of its 128 rows of a k-block (and multicasts it).
        if (!encode_2d(&ta, A, M, K, lda, pl.v->info.pair == 2 ? kBM / 2 : kBM)) return GEMMPIPE_ERR_INTERNAL;
        const int per_mma = pl.v->info.BN / (pl.v->info.BN > 256 ? pl.v->info.BN / 256 : 1) / 2 / 64;
        const int bk = pl.v->info.BK;
        b_groups = pl.v->info.pair && N % 64 == 0 && encode_b_groups(&tb, B, K, N, ldb, bk, per_mma) ? 1 : 0;
        if (!b_groups && !encode_2d(&tb, B, K, N, ldb, bk)) return GEMMPIPE_ERR_INTERNAL;
    }
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.A = A;
    p.lda = lda;
    p.B = B;
    p.ldb = ldb;
    p.C = C;
    p.ldc = ldc;
    set_schedule(pl, dev, s, p);
    p.b_groups = b_groups;
    p.tma_store = pl.vec_store && encode_c(&tc, C, M, N, ldc, pl.v->info.int_out != 0) ? 1 : 0;
    p.stall_kb = -1;
    p.timeout_ns = 2000000000ull + static_cast<uint64_t>(pl.kb_per_chunk) * 10000ull;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_stall.kb >= 0) {
            p.stall_kb = g_stall.kb;
            p.timeout_ns = static_cast<uint64_t>(g_stall.timeout_ms) * 1000000ull;
            g_stall = StallHook();
        }
        if (g_trace_hook.buf) {
            const Variant *tv = traced_twin(pl.v);
            if (tv) {
                pl.v = tv;
                p.trace = g_trace_hook.buf;
                p.trace_n = g_trace_hook.n;
            }
            g_trace_hook = TraceHook();
        }
    }
    if (gp::status_word(&p.status) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_LAUNCH;
    }
    TimedRegion tr(true, s);
    const cudaError_t e = pl.v->launch(ta, tb, tc, p, pl.grid, s);
    tr.end();
    if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    return GEMMPIPE_OK;
}

gemmpipe_status_t zero_c(void *C, int64_t bytes, const DeviceInfo &d, cudaStream_t s)
{
    TimedRegion tr(false, s);
    const cudaError_t e = gp::launch_zero_fill(C, bytes, d.sms, s);
    tr.end();
    if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    return GEMMPIPE_OK;
}

int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

// TMA can describe a row-major fp16 operand whose base and row pitch are
// multiples of 16 bytes.
bool operand_tma_ok(const void *p, int64_t ld) { return aligned16(p) && (ld * 2) % 16 == 0; }

// Misaligned fp16 operands are padded unless the bounded-load producer is forced.
bool pad_wanted(const void *A, int64_t K, const void *B, int64_t N)
{
    if (operand_tma_ok(A, K) && operand_tma_ok(B, N)) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_override.producer != 1;
}

// Pads one or two operands (rows1 == 0: one) in a single launch.
gemmpipe_status_t pad_operands(const uint16_t *src0, int64_t rows0, int64_t cols0, uint16_t *dst0, int64_t pitch0,
                               const uint16_t *src1, int64_t rows1, int64_t cols1, uint16_t *dst1, int64_t pitch1,
                               const DeviceInfo &d, cudaStream_t s)
{
    TimedRegion tr(false, s);
    const cudaError_t e =
        gp::launch_pad_f16(src0, rows0, cols0, dst0, pitch0, src1, rows1, cols1, dst1, pitch1, d.sms, s);
    tr.end();
    if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    return GEMMPIPE_OK;
}

int64_t s8_workspace_bytes(int64_t M, int64_t N, int64_t K) { return 2 * (M * round8(K) + K * round8(N)); }

}  // namespace

namespace gp {

// The INT8 flow of gemm_s8s8s32 with caller-provided scratch for the fp16
// copies: no workspace allocation and no timing events.  Used only by
// gemm_s8s8s32_noalloc.
gemmpipe_status_t s8_check_fixed_scratch(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B,
                                         const int32_t *C, int64_t scratch_bytes)
{
    const gemmpipe_status_t st = check_shape(M, N, K, A, B, C, 1, 4);
    if (st != GEMMPIPE_OK) return st;
    if (M == 0 || N == 0 || K == 0) return GEMMPIPE_OK;
    return s8_workspace_bytes(M, N, K) <= scratch_bytes ? GEMMPIPE_OK : GEMMPIPE_ERR_INVALID_VALUE;
}

gemmpipe_status_t s8_with_fixed_scratch(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B,
                                        int32_t *C, cudaStream_t s, uint16_t *scratch, int64_t scratch_bytes)
{
    gemmpipe_status_t st = s8_check_fixed_scratch(M, N, K, A, B, C, scratch_bytes);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    DeviceInfo d;
    if ((st = device_info(&d, nullptr)) != GEMMPIPE_OK) return st;
    if ((st = check_device_pointers(K, A, B, C, 1, 4)) != GEMMPIPE_OK) return st;
    if (K == 0) {
        if (gp::launch_zero_fill(C, M * N * 4, d.sms, s) != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
        g_launches.fetch_add(1);
        return GEMMPIPE_OK;
    }
    const int64_t Kp = round8(K), Np = round8(N);
    uint16_t *A16 = scratch;
    uint16_t *B16 = scratch + M * Kp;
    if (gp::launch_widen_s8_f16(A, M, K, A16, Kp, B, K, N, B16, Np, d.sms, s) != cudaSuccess)
        return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    Plan pl;
    // Whole tiles only: split tiles would need a partial-sum workspace.
    if ((st = make_plan(true, M, N, K, A16, Kp, B16, Np, C, N, d, &pl, false, false)) != GEMMPIPE_OK) return st;
    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (!encode_2d(&ta, A16, M, K, Kp, pl.v->info.pair == 2 ? kBM / 2 : kBM) ||
        !encode_2d(&tb, B16, K, N, Np, pl.v->info.BK))
        return GEMMPIPE_ERR_INTERNAL;
    GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.A = A16;
    p.lda = Kp;
    p.B = B16;
    p.ldb = Np;
    p.C = C;
    p.ldc = N;
    p.m_tiles = pl.m_tiles;
    p.tiles = pl.tiles;
    p.group_m = pl.group_m;
    p.units = pl.units;
    p.dp_tiles = pl.dp_tiles;
    p.sk_work = 0;
    p.epoch = 0;
    p.partials = nullptr;
    p.flags = nullptr;
    p.num_kb = pl.num_kb;
    p.kb_per_chunk = pl.kb_per_chunk;
    p.vec_store = pl.vec_store;
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    p.tma_store = pl.vec_store && encode_c(&tc, C, M, N, N, true) ? 1 : 0;
    p.stall_kb = -1;
    p.timeout_ns = 2000000000ull + static_cast<uint64_t>(pl.kb_per_chunk) * 10000ull;
    if (gp::status_word(&p.status) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_LAUNCH;
    }
    if (pl.v->launch(ta, tb, tc, p, pl.grid, s) != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    return GEMMPIPE_OK;
}

}  // namespace gp

namespace {

// ------------------------------------------------------- host-buffer calls

// Side streams and events of the host-buffer entry points, per (device,
// caller stream): copies to the device run on `in`, copies back on `out`,
// kernels on the caller's stream; events order the three.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    std::vector<cudaEvent_t> ev;
};
std::map<std::pair<int, cudaStream_t>, HostPipe> g_host;

gemmpipe_status_t host_pipe(int dev, cudaStream_t s, size_t events, HostPipe *out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    HostPipe &h = g_host[std::make_pair(dev, s)];
    if (!h.in && cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        h.in = nullptr;
        return GEMMPIPE_ERR_LAUNCH;
    }
    if (!h.out && cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        h.out = nullptr;
        return GEMMPIPE_ERR_LAUNCH;
    }
    while (h.ev.size() < events) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return GEMMPIPE_ERR_LAUNCH;
        }
        h.ev.push_back(e);
    }
    *out = h;
    return GEMMPIPE_OK;
}

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// One host-buffer call: B and the row panels of A go to device buffers on
// the `in` stream, panel p's GEMM runs on the caller's stream once its rows
// have arrived, and its rows of C go back on the `out` stream while later
// panels compute.  With `parts` > 1 the first panel is computed in two
// column halves: B comes in those halves (the first panel's rows of A before
// them), so the first C values start back after half of B instead of all
// of it.  `prep_b(c0, nc)` enqueues what B's columns [c0, c0 + nc) need once
// they have arrived; `panel(r0, mp, c0, nc)` enqueues the kernels of C's rows
// [r0, r0 + mp) x columns [c0, c0 + nc).  Everything is enqueued before the
// first copy back, so a pageable C (whose copies return only when done)
// still overlaps the remaining panels.
template <class PrepFn, class PanelFn>
gemmpipe_status_t host_call(int dev, cudaStream_t s, int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                            void *C, int ab_bytes, int c_bytes, void *dA, void *dB, void *dC, int parts,
                            PrepFn prep_b, PanelFn panel)
{
    const int64_t rows = gemmpipe_host_panel_rows(M);
    const int64_t P = (M + rows - 1) / rows;
    const int Q = K > 0 && parts > 1 ? 2 : 1;  // column parts of the first panel: one or two (halves)
    const int64_t w = Q > 1 ? N / Q / 16 * 16 : N;   // whole 16-column groups: bases stay on 16 bytes
    const auto col0 = [&](int q) { return q * w; };
    const auto ncol = [&](int q) { return q == Q - 1 ? N - col0(q) : w; };
    HostPipe h;
    gemmpipe_status_t st = host_pipe(dev, s, static_cast<size_t>(2 * Q + 2 * P + 3), &h);
    if (st != GEMMPIPE_OK) return st;
    // Events: [0] start; ev_b[q] B's part q in; ev_a[p] A's panel p in;
    // ev_h[q] the first panel's part q done; ev_c[p] panel p done (p >= 1);
    // ev_end[0] all in, ev_end[1] all out.
    cudaEvent_t *ev = h.ev.data();
    cudaEvent_t *ev_b = ev + 1, *ev_a = ev_b + Q, *ev_h = ev_a + P, *ev_c = ev_h + Q, *ev_end = ev_c + P;
    const auto ok = [](cudaError_t e) {
        if (e == cudaSuccess) return true;
        cudaGetLastError();
        return false;
    };
    if (!ok(cudaEventRecord(ev[0], s)) || !ok(cudaStreamWaitEvent(h.in, ev[0], 0)) ||
        !ok(cudaStreamWaitEvent(h.out, ev[0], 0)))
        return GEMMPIPE_ERR_LAUNCH;
    const char *hA = static_cast<const char *>(A);
    const char *hB = static_cast<const char *>(B);
    char *dAc = static_cast<char *>(dA);
    char *dBc = static_cast<char *>(dB);
    char *dCc = static_cast<char *>(dC);
    char *hC = static_cast<char *>(C);
    const size_t brow = static_cast<size_t>(N * ab_bytes), crow = static_cast<size_t>(N * c_bytes);
    auto rows_of = [&](int64_t p) { return M - p * rows < rows ? M - p * rows : rows; };
    auto copy_a = [&](int64_t p) {
        const int64_t r0 = p * rows;
        return ok(cudaMemcpyAsync(dAc + r0 * K * ab_bytes, hA + r0 * K * ab_bytes,
                                  static_cast<size_t>(rows_of(p) * K * ab_bytes), cudaMemcpyDefault, h.in)) &&
               ok(cudaEventRecord(ev_a[p], h.in));
    };
    // B's columns [c0, c0 + nc) in, as a 2-D copy (whole rows: one copy).
    auto copy_b = [&](int64_t c0, int64_t nc) {
        if (nc == N)
            return ok(cudaMemcpyAsync(dB, B, static_cast<size_t>(K) * brow, cudaMemcpyDefault, h.in));
        return ok(cudaMemcpy2DAsync(dBc + c0 * ab_bytes, brow, hB + c0 * ab_bytes, brow,
                                    static_cast<size_t>(nc * ab_bytes), static_cast<size_t>(K), cudaMemcpyDefault,
                                    h.in));
    };
    bool good = true;
    if (K > 0) {
        if (Q > 1) good = copy_a(0);
        for (int q = 0; good && q < Q; ++q) good = copy_b(col0(q), ncol(q)) && ok(cudaEventRecord(ev_b[q], h.in));
        for (int64_t p = Q > 1 ? 1 : 0; good && p < P; ++p) good = copy_a(p);
    }
    auto wait = [&](cudaEvent_t e) { return K == 0 || ok(cudaStreamWaitEvent(s, e, 0)); };
    if (good) good = wait(ev_a[0]);
    for (int q = 0; good && st == GEMMPIPE_OK && q < Q; ++q) {
        good = wait(ev_b[q]);
        if (good && (st = prep_b(col0(q), ncol(q))) == GEMMPIPE_OK &&
            (st = panel(0, rows_of(0), col0(q), ncol(q))) == GEMMPIPE_OK)
            good = ok(cudaEventRecord(ev_h[q], s));
    }
    for (int64_t p = 1; good && st == GEMMPIPE_OK && p < P; ++p) {
        good = wait(ev_a[p]);
        if (good && (st = panel(p * rows, rows_of(p), 0, N)) == GEMMPIPE_OK) good = ok(cudaEventRecord(ev_c[p], s));
    }
    if (good && st == GEMMPIPE_OK) {
        const size_t r = static_cast<size_t>(rows_of(0));
        for (int q = 0; good && q < Q; ++q) {
            good = ok(cudaStreamWaitEvent(h.out, ev_h[q], 0));
            if (good && Q == 1)
                good = ok(cudaMemcpyAsync(hC, dCc, r * crow, cudaMemcpyDefault, h.out));
            else if (good)
                good = ok(cudaMemcpy2DAsync(hC + col0(q) * c_bytes, crow, dCc + col0(q) * c_bytes, crow,
                                            static_cast<size_t>(ncol(q) * c_bytes), r, cudaMemcpyDefault, h.out));
        }
        for (int64_t p = 1; good && p < P; ++p) {
            const int64_t r0 = p * rows;
            good = ok(cudaStreamWaitEvent(h.out, ev_c[p], 0)) &&
                   ok(cudaMemcpyAsync(hC + r0 * crow, dCc + r0 * crow, static_cast<size_t>(rows_of(p)) * crow,
                                      cudaMemcpyDefault, h.out));
        }
    }
    // Whatever was enqueued, the caller's stream ends after both side
    // streams, so later work on it never races these copies.
    const bool joined = ok(cudaEventRecord(ev_end[0], h.in)) && ok(cudaEventRecord(ev_end[1], h.out)) &&
                        ok(cudaStreamWaitEvent(s, ev_end[0], 0)) && ok(cudaStreamWaitEvent(s, ev_end[1], 0));
    if (st != GEMMPIPE_OK) return st;
    return good && joined ? GEMMPIPE_OK : GEMMPIPE_ERR_LAUNCH;
}

// Column parts of the first panel: two (halves) when B holds at least 4 MiB
// and N is a multiple of 32, else one; parts are whole 16-column groups, so
// every TMA base and pitch stays on 16 bytes.  End to end at 4096^3 (four
// panels), INT8 / FP16: 523 / 628 us in one part, 491 / 592 us in halves,
// 500 / 615 us in quarters -- more, smaller copies cost more than the
// earlier start saves.
int host_col_parts(int64_t N, int64_t K, int ab_bytes)
{
    const int64_t b = K * N * ab_bytes;
    if (N % 32 == 0 && N >= 512 && b >= (int64_t(4) << 20)) return 2;
    return 1;
}

// Device buffers of a host-buffer call: A, B and C, each 256-byte aligned.
gemmpipe_status_t host_buffers(int dev, cudaStream_t s, int64_t M, int64_t N, int64_t K, int ab_bytes, int c_bytes,
                               void **dA, void **dB, void **dC)
{
    const int64_t a = align256(M * K * ab_bytes), b = align256(K * N * ab_bytes), c = M * N * c_bytes;
    void *ws = nullptr;
    gemmpipe_status_t st = workspace(dev, s, a + b + c, &ws, kWsHost);
    if (st != GEMMPIPE_OK) return st;
    *dA = ws;
    *dB = static_cast<char *>(ws) + a;
    *dC = static_cast<char *>(ws) + a + b;
    return GEMMPIPE_OK;
}

}  // namespace

extern "C" {

int64_t gemmpipe_host_panel_rows(int64_t M)
{
    if (M <= 0) return 512;
    // A quarter of M: fewer, larger copies beat finer overlap on this link
    // (INT8 4096^3: 491 us with 4 panels, 506 with 8, 635 with 16).
    int64_t r = (M + 3) / 4;
    r = (r + 255) / 256 * 256;
    return r < 512 ? 512 : r;
}

gemmpipe_status_t gemm_s8s8s32_host(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B, int32_t *C,
                                    gemmpipe_stream_t stream)
{
    gemmpipe_status_t st = check_shape(M, N, K, A, B, C, 1, 4);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceInfo d;
    if ((st = device_info(&d, &dev)) != GEMMPIPE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    if ((st = host_buffers(dev, s, M, N, K, 1, 4, &dA, &dB, &dC)) != GEMMPIPE_OK) return st;
    const int8_t *A8 = static_cast<const int8_t *>(dA), *B8 = static_cast<const int8_t *>(dB);
    int32_t *C32 = static_cast<int32_t *>(dC);
    // B is widened once; each panel widens its rows of A into their place
    // in the operand workspace and runs the GEMM on them.  Plans that do not
    // use widened copies (the comparison path, in-kernel widening) and K = 0
    // go through gemm_s8s8s32 per panel.
    const bool direct = K == 0 || imma_wanted(A8, K) || s8_convert_ok(A8, K, B8, N);
    const int64_t Kp = round8(K), Np = round8(N);
    uint16_t *A16 = nullptr, *B16 = nullptr;
    if (!direct) {
        void *ws = nullptr;
        if ((st = workspace(dev, s, s8_workspace_bytes(M, N, K), &ws)) != GEMMPIPE_OK) return st;
        A16 = static_cast<uint16_t *>(ws);
        B16 = A16 + M * Kp;
    }
    auto launched = [&](cudaError_t e) {
        if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
        g_launches.fetch_add(1);
        return GEMMPIPE_OK;
    };
    // B's columns [c0, c0 + nc) into their place in the fp16 copy.
    auto prep_b = [&](int64_t c0, int64_t nc) {
        if (direct) return GEMMPIPE_OK;
        TimedRegion tr(false, s);
        const cudaError_t e =
            nc == N ? gp::launch_widen_s8_f16(B8, K, N, B16, Np, B8, 0, N, B16, Np, d.sms, s)
                    : gp::launch_widen_s8_f16_cols(B8 + c0, K, nc, N, B16 + c0, Np, d.sms, s);
        tr.end();
        return launched(e);
    };
    const int parts = direct ? 1 : host_col_parts(N, K, 1);
    return host_call(dev, s, M, N, K, A, B, C, 1, 4, dA, dB, dC, parts, prep_b,
                     [&](int64_t r0, int64_t mp, int64_t c0, int64_t nc) {
        if (direct) return gemm_s8s8s32(mp, N, K, A8 + r0 * K, B8, C32 + r0 * N, stream);
        gemmpipe_status_t e;
        if (c0 == 0) {  // the panel's rows of A, once
            TimedRegion tr(false, s);
            const cudaError_t ce = gp::launch_widen_s8_f16(A8 + r0 * K, mp, K, A16 + r0 * Kp, Kp, A8 + r0 * K, 0, K,
                                                           A16 + r0 * Kp, Kp, d.sms, s);
            tr.end();
            if ((e = launched(ce)) != GEMMPIPE_OK) return e;
        }
        Plan pl;
        if ((e = make_plan(true, mp, nc, K, A16 + r0 * Kp, Kp, B16 + c0, Np, C32 + r0 * N + c0, N, d, &pl)) !=
            GEMMPIPE_OK)
            return e;
        return run_plan(pl, dev, mp, nc, K, A16 + r0 * Kp, Kp, B16 + c0, Np, C32 + r0 * N + c0, N, s);
    });
}

gemmpipe_status_t gemm_f16f32_host(int64_t M, int64_t N, int64_t K, const gemmpipe_half_t *A,
                                   const gemmpipe_half_t *B, float *C, gemmpipe_stream_t stream)
{
    gemmpipe_status_t st = check_shape(M, N, K, A, B, C, 2, 4);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceInfo d;
    if ((st = device_info(&d, &dev)) != GEMMPIPE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    if ((st = host_buffers(dev, s, M, N, K, 2, 4, &dA, &dB, &dC)) != GEMMPIPE_OK) return st;
    const gemmpipe_half_t *A16 = static_cast<const gemmpipe_half_t *>(dA);
    const gemmpipe_half_t *B16 = static_cast<const gemmpipe_half_t *>(dB);
    float *C32 = static_cast<float *>(dC);
    // The first panel's column parts run as plans on B's column slices,
    // which needs TMA-describable operands (K a multiple of 8).
    const int parts = K % 8 == 0 ? host_col_parts(N, K, 2) : 1;
    return host_call(dev, s, M, N, K, A, B, C, 2, 4, dA, dB, dC, parts,
                     [](int64_t, int64_t) { return GEMMPIPE_OK; },
                     [&](int64_t r0, int64_t mp, int64_t c0, int64_t nc) {
        if (nc == N) return gemm_f16f32(mp, N, K, A16 + r0 * K, B16, C32 + r0 * N, stream);
        Plan pl;
        gemmpipe_status_t e;
        const uint16_t *a = A16 + r0 * K, *b = B16 + c0;
        if ((e = make_plan(false, mp, nc, K, a, K, b, N, C32 + r0 * N + c0, N, d, &pl)) != GEMMPIPE_OK) return e;
        return run_plan(pl, dev, mp, nc, K, a, K, b, N, C32 + r0 * N + c0, N, s);
    });
}


gemmpipe_status_t gemm_f16f32(int64_t M, int64_t N, int64_t K, const gemmpipe_half_t *A, const gemmpipe_half_t *B,
                              float *C, gemmpipe_stream_t stream)
{
    gemmpipe_status_t st = check_shape(M, N, K, A, B, C, 2, 4);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    DeviceInfo d;
    int dev = 0;
    if ((st = device_info(&d, &dev)) != GEMMPIPE_OK) return st;
    if ((st = check_device_pointers(K, A, B, C, 2, 4)) != GEMMPIPE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return zero_c(C, M * N * 4, d, s);
    const uint16_t *Ause = A, *Buse = B;
    int64_t lda = K, ldb = N;
    if (pad_wanted(A, K, B, N)) {
        // "Pad the matrices" remedy: aligned copies in the stream's workspace,
        // then the TMA producer.  Without a workspace the bounded-load
        // producer reads the original operands instead.
        const bool pa = !operand_tma_ok(A, K), pb = !operand_tma_ok(B, N);
        const int64_t Kp = round8(K), Np = round8(N);
        const int64_t bytes = (pa ? 2 * M * Kp : 0) + (pb ? 2 * K * Np : 0);
        void *ws = nullptr;
        if (workspace(dev, s, bytes, &ws) == GEMMPIPE_OK) {
            uint16_t *w = static_cast<uint16_t *>(ws);
            uint16_t *wa = pa ? w : nullptr;
            uint16_t *wb = pb ? w + (pa ? M * Kp : 0) : nullptr;
            if (pa && pb)
                st = pad_operands(A, M, K, wa, Kp, B, K, N, wb, Np, d, s);
            else if (pa)
                st = pad_operands(A, M, K, wa, Kp, nullptr, 0, 0, nullptr, 0, d, s);
            else
                st = pad_operands(B, K, N, wb, Np, nullptr, 0, 0, nullptr, 0, d, s);
            if (st != GEMMPIPE_OK) return st;
            if (pa) {
                Ause = wa;
                lda = Kp;
            }
            if (pb) {
                Buse = wb;
                ldb = Np;
            }
        }
    }
    Plan pl;
    if ((st = make_plan(false, M, N, K, Ause, lda, Buse, ldb, C, N, d, &pl)) != GEMMPIPE_OK) return st;
    return run_plan(pl, dev, M, N, K, Ause, lda, Buse, ldb, C, N, s);
}

gemmpipe_status_t gemm_s8s8s32(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B, int32_t *C,
                               gemmpipe_stream_t stream)
{
    gemmpipe_status_t st = check_shape(M, N, K, A, B, C, 1, 4);
    if (st != GEMMPIPE_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceInfo d;
    if ((st = device_info(&d, &dev)) != GEMMPIPE_OK) return st;
    if ((st = check_device_pointers(K, A, B, C, 1, 4)) != GEMMPIPE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return zero_c(C, M * N * 4, d, s);
    if (imma_wanted(A, K)) {
        // Comparison path: B transposed, then warp-level integer MMA.
        const int64_t ldbt = gp::imma_bt_pitch(K);
        void *ws = nullptr;
        if ((st = workspace(dev, s, imma_workspace_bytes(N, K), &ws)) != GEMMPIPE_OK) return st;
        int8_t *BT = static_cast<int8_t *>(ws);
        {
            TimedRegion tr(false, s);
            const cudaError_t e = gp::launch_transpose_s8(B, K, N, BT, ldbt, s);
            tr.end();
            if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
            g_launches.fetch_add(1);
        }
        TimedRegion tr(true, s);
        int stages = 0;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            stages = g_override.stages;
        }
        const cudaError_t e = gp::launch_imma_s8(A, BT, ldbt, C, M, N, K, stages, s);
        tr.end();
        if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
        g_launches.fetch_add(1);
        return GEMMPIPE_OK;
    }
    if (s8_convert_ok(A, K, B, N)) {
        // int8 tiles straight from A and B, widened inside the kernel.
        Plan pl;
        const uint16_t *A8 = reinterpret_cast<const uint16_t *>(A);
        const uint16_t *B8 = reinterpret_cast<const uint16_t *>(B);
        if ((st = make_plan(true, M, N, K, A8, K, B8, N, C, N, d, &pl, true)) != GEMMPIPE_OK) return st;
        return run_plan(pl, dev, M, N, K, A8, K, B8, N, C, N, s);
    }
    const int64_t Kp = round8(K), Np = round8(N);
    void *ws = nullptr;
    if ((st = workspace(dev, s, s8_workspace_bytes(M, N, K), &ws)) != GEMMPIPE_OK) return st;
    uint16_t *A16 = static_cast<uint16_t *>(ws);
    uint16_t *B16 = A16 + M * Kp;
    {
        TimedRegion tr(false, s);
        const cudaError_t e = gp::launch_widen_s8_f16(A, M, K, A16, Kp, B, K, N, B16, Np, d.sms, s);
        tr.end();
        if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
        g_launches.fetch_add(1);
    }
    Plan pl;
    if ((st = make_plan(true, M, N, K, A16, Kp, B16, Np, C, N, d, &pl)) != GEMMPIPE_OK) return st;
    return run_plan(pl, dev, M, N, K, A16, Kp, B16, Np, C, N, s);
}

gemmpipe_status_t gemmpipe_get_device_status(gemmpipe_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_LAUNCH;
    }
    int *w = nullptr;
    if (gp::status_word(&w) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_LAUNCH;
    }
    int v = 0;
    if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMMPIPE_ERR_LAUNCH;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    }
    if (v == GEMMPIPE_ERR_TIMEOUT) return GEMMPIPE_ERR_TIMEOUT;
    if (v != 0) return GEMMPIPE_ERR_INTERNAL;
    return GEMMPIPE_OK;
}

const char *gemmpipe_status_string(gemmpipe_status_t status)
{
    switch (status) {
    case GEMMPIPE_OK: return "ok";
    case GEMMPIPE_ERR_INVALID_VALUE: return "invalid value";
    case GEMMPIPE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case GEMMPIPE_ERR_LAUNCH: return "kernel launch or CUDA runtime error";
    case GEMMPIPE_ERR_TIMEOUT: return "a pipeline wait on the device ran out of time";
    case GEMMPIPE_ERR_INTERNAL: return "internal error";
    case GEMMPIPE_ERR_OUT_OF_MEMORY: return "out of device memory";
    }
    return "unknown status";
}

double gemmpipe_compute_load_ratio(int BM, int BN, int BK, int elem_bytes)
{
    if (BM < 1 || BN < 1 || BK < 1 || elem_bytes < 1) return -1.0;
    const double mac_flops = 2.0 * BM * static_cast<double>(BN) * BK;
    const double tile_bytes = (static_cast<double>(BM) * BK + static_cast<double>(BK) * BN) * elem_bytes;
    return mac_flops / tile_bytes;
}

int64_t gemmpipe_stage_smem_bytes(int BM, int BN, int BK, int elem_bytes, int stages)
{
    if (BM < 1 || BN < 1 || BK < 1 || elem_bytes < 1 || stages < 1) return -1;
    return static_cast<int64_t>(stages) * (static_cast<int64_t>(BM) * BK + static_cast<int64_t>(BK) * BN) *
           elem_bytes;
}

gemmpipe_status_t gemmpipe_plan(int dtype, int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                                const void *C, gemmpipe_plan_t *plan)
{
    if (!plan || (dtype != 0 && dtype != 1)) return GEMMPIPE_ERR_INVALID_VALUE;
    const bool s8 = dtype == 0;
    static const uint16_t *const kAligned = reinterpret_cast<const uint16_t *>(256);
    if (!A) A = kAligned;
    if (!B) B = kAligned;
    if (!C) C = kAligned;
    gemmpipe_status_t st = check_shape(M, N, K, A, B, C, s8 ? 1 : 2, 4);
    if (st != GEMMPIPE_OK) return st;
    DeviceInfo d;
    if ((st = device_info(&d, nullptr)) != GEMMPIPE_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    if (M == 0 || N == 0 || K == 0) return GEMMPIPE_OK;
    Plan pl;
    if (s8 && imma_wanted(static_cast<const int8_t *>(A), K)) {
        gp::VariantInfo f;
        int stages = 0;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            stages = g_override.stages;
        }
        gp::imma_plan_info(&f, stages);
        plan->producer = f.producer;
        plan->BM = f.BM;
        plan->BN = f.BN;
        plan->BK = f.BK;
        plan->stages = f.stages;
        plan->k_chunk = static_cast<int>(K);
        plan->threads = f.threads;
        plan->tiles = ((M + f.BM - 1) / f.BM) * ((N + f.BN - 1) / f.BN);
        plan->grid = static_cast<int>(plan->tiles);
        plan->units = plan->tiles;
        plan->k_blocks = (K + f.BK - 1) / f.BK;
        plan->smem_bytes = f.smem_bytes;
        plan->vector_store = 0;
        plan->operand_copy = 3;
        plan->workspace_bytes = imma_workspace_bytes(N, K);
        return GEMMPIPE_OK;
    }
    if (s8 && s8_convert_ok(A, K, B, N)) {
        st = make_plan(true, M, N, K, A, K, B, N, C, N, d, &pl, true);
    } else if (s8) {
        // The widened copies are 16-byte aligned with 16-byte row pitches.
        st = make_plan(true, M, N, K, kAligned, round8(K), kAligned, round8(N), C, N, d, &pl);
        plan->workspace_bytes = s8_workspace_bytes(M, N, K);
        plan->operand_copy = 1;
    } else if (pad_wanted(A, K, B, N)) {
        const bool pa = !operand_tma_ok(A, K), pb = !operand_tma_ok(B, N);
        st = make_plan(false, M, N, K, pa ? kAligned : A, pa ? round8(K) : K, pb ? kAligned : B,
                       pb ? round8(N) : N, C, N, d, &pl);
        plan->workspace_bytes = (pa ? 2 * M * round8(K) : 0) + (pb ? 2 * K * round8(N) : 0);
        plan->operand_copy = 2;
    } else {
        st = make_plan(false, M, N, K, A, K, B, N, C, N, d, &pl);
    }
    if (st != GEMMPIPE_OK) return st;
    const gp::VariantInfo &f = pl.v->info;
    plan->producer = f.producer;
    plan->BM = f.pair ? 2 * f.BM : f.BM;
    plan->cta_pair = f.pair;
    plan->BN = f.pair == 2 ? 2 * f.BN : f.BN;  // a quad's tile is two pairs' tiles wide
    plan->BK = f.BK;
    plan->stages = f.stages;
    plan->k_chunk = static_cast<int>(pl.kb_per_chunk * f.BK < K ? pl.kb_per_chunk * f.BK : K);
    plan->threads = f.threads;
    plan->grid = pl.grid;
    plan->tiles = pl.tiles;
    plan->units = pl.units;
    plan->split_tiles = pl.sk_tiles;
    plan->k_blocks = pl.num_kb;
    plan->smem_bytes = f.smem_bytes;
    plan->vector_store = pl.vec_store;
    plan->workspace_bytes += pl.split_bytes();

    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_set_plan_override(int producer, int bn, int stages, int cta_pair, int split)
{
    if (producer < -1 || producer > 2) return GEMMPIPE_ERR_INVALID_VALUE;
    if (bn != 0 && bn != 128 && bn != 256 && bn != 512) return GEMMPIPE_ERR_INVALID_VALUE;
    if (stages < 0 || stages > 16) return GEMMPIPE_ERR_INVALID_VALUE;
    if (cta_pair < -1 || cta_pair > 2) return GEMMPIPE_ERR_INVALID_VALUE;
    if (split < -1 || split > 1) return GEMMPIPE_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_override.producer = producer;
    g_override.bn = bn;
    g_override.stages = stages;
    g_override.pair = cta_pair;
    g_override.split = split;
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_set_plan_bk(int bk)
{
    if (bk != 0 && bk != 64 && bk != 128) return GEMMPIPE_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_override.bk = bk;
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_release_workspaces(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    const bool have = cudaGetDevice(&cur) == cudaSuccess;
    for (auto &kv : g_ws) {
        if (kv.second.ptr) {
            cudaSetDevice(std::get<0>(kv.first));
            cudaFree(kv.second.ptr);
        }
    }
    g_ws.clear();
    for (auto &kv : g_host) {
        cudaSetDevice(kv.first.first);
        if (kv.second.in) cudaStreamDestroy(kv.second.in);
        if (kv.second.out) cudaStreamDestroy(kv.second.out);
        for (cudaEvent_t e : kv.second.ev) cudaEventDestroy(e);
    }
    g_host.clear();
    if (have) cudaSetDevice(cur);
    cudaGetLastError();
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_timing_enable(int enable)
{
    std::lock_guard<std::mutex> lk(g_mu);
    g_timing.enabled = enable != 0;
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_timing_read(double *gemm_ms, int64_t *gemm_launches, double *aux_ms,
                                       int64_t *aux_launches)
{
    std::lock_guard<std::mutex> lk(g_mu);
    gemmpipe_status_t st = GEMMPIPE_OK;
    auto sum = [&](std::vector<std::pair<cudaEvent_t, cudaEvent_t>> &v, double *ms, int64_t *n) {
        double t = 0.0;
        for (auto &pr : v) {
            float f = 0.f;
            if (cudaEventSynchronize(pr.second) != cudaSuccess ||
                cudaEventElapsedTime(&f, pr.first, pr.second) != cudaSuccess) {
                cudaGetLastError();
                st = GEMMPIPE_ERR_LAUNCH;
            }
            t += f;
            g_timing.pool.push_back(pr.first);
            g_timing.pool.push_back(pr.second);
        }
        if (ms) *ms = t;
        if (n) *n = static_cast<int64_t>(v.size());
        v.clear();
    };
    sum(g_timing.gemm, gemm_ms, gemm_launches);
    sum(g_timing.aux, aux_ms, aux_launches);
    return st;
}

int64_t gemmpipe_launch_count(void) { return g_launches.load(); }

gemmpipe_status_t gemmpipe_copy(void *dst, const void *src, int64_t bytes, gemmpipe_stream_t stream)
{
    if (bytes < 0) return GEMMPIPE_ERR_INVALID_VALUE;
    if (bytes == 0) return GEMMPIPE_OK;
    if (!dst || !src) return GEMMPIPE_ERR_INVALID_VALUE;
    DeviceInfo d;
    gemmpipe_status_t st = device_info(&d, nullptr);
    if (st != GEMMPIPE_OK) return st;
    if ((st = check_pointer(dst, 1)) != GEMMPIPE_OK || (st = check_pointer(src, 1)) != GEMMPIPE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    TimedRegion tr(false, s);
    const cudaError_t e = gp::launch_copy(dst, src, bytes, d.sms, s);
    tr.end();
    if (e != cudaSuccess) return GEMMPIPE_ERR_LAUNCH;
    g_launches.fetch_add(1);
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_test_trace(void *buffer, int64_t entries)
{
    if (entries < 0 || entries > (int64_t(1) << 20)) return GEMMPIPE_ERR_INVALID_VALUE;
    if (entries == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        g_trace_hook = TraceHook();
        return GEMMPIPE_OK;
    }
    gemmpipe_status_t st = check_pointer(buffer, 8);
    if (st != GEMMPIPE_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    g_trace_hook.buf = static_cast<unsigned long long *>(buffer);
    g_trace_hook.n = entries;
    return GEMMPIPE_OK;
}

gemmpipe_status_t gemmpipe_test_inject_stall(int64_t k_block, int timeout_ms)
{
    if (k_block >= 0 && (timeout_ms < 1 || timeout_ms > 60000)) return GEMMPIPE_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_stall.kb = k_block < 0 ? -1 : k_block;
    g_stall.timeout_ms = timeout_ms;
    return GEMMPIPE_OK;
}

}  // extern "C"
