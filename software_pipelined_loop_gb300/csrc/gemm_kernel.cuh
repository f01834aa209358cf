// gemm_kernel.cuh -- the software-pipelined tiled GEMM C = A * B for sm_103a.
//
// "Pipeline GPU Kernel" (skill page), Steps 3-4, turns a sequential
// load / sync / compute / sync K loop into a prologue, a main loop that loads
// K-tile n+1 while the tensor cores work on K-tile n, and an epilogue that
// computes the last tile, with two shared-memory buffers used alternately.
// Here the same schedule is spread over warps with separate jobs and the
// double buffer becomes an S-stage ring guarded by mbarriers:
//
//   producer  (1 warp issuing TMA tile loads, or 8 warps doing
//             bounds-checked loads into registers and shared-memory stores --
//             the page's LDG-register variant, used when TMA cannot describe
//             the input) waits empty[s], fills stage s with the A tile
//             (BM x BK) and the B tile (BK x BN) of k-block kb, and signals
//             full[s];
//   issuer    (1 warp) waits full[s], issues BK/16 tcgen05.mma (K = 16;
//             M = 256 over a CTA pair with cta_group::2, else 128) into a
//             TMEM accumulator, then tcgen05.commit -> empty[s] returns the
//             stage to the producer as soon as the tensor cores have read it;
//   epilogue  (8 warps) waits tfull[b], copies the accumulator to registers
//             with tcgen05.ld, frees it, and stores C through a per-warp
//             staging tile (one TMA store per 32 x 32 block, or
//             row-contiguous masked stores).
//
// The TMA producer and the issuer run their loops on the whole warp, one
// elected lane issuing the copies, MMAs and commits: the loop state and the
// descriptors stay warp-uniform, and the coupled ring keeps the tensor pipe
// fed (with a single thread per role, the same pipeline ran ~25% slower).
//
// The page's prologue is the producer running up to S stages ahead; its
// "compute the last tile" epilogue is the issuer's final commit on tfull.
// Two TMEM accumulators let tile t+1's MMAs run while tile t is stored.
//
// The CTAs are persistent (one per SM, or one pair per two SMs) and walk a
// static schedule (WorkIter): whole tiles round-robin, then equal ranges of
// the split tiles' k-blocks (stream-K), whose partial sums meet in a
// workspace.  TMA variants run 12 warps: warps 0-3 (producer, issuer, two
// idle) give registers to the two epilogue warpgroups with setmaxnreg.
//
// For the INT8 path (operands widened to fp16, see the C header) an
// accumulator covers at most `kb_per_chunk` k-blocks; the epilogue turns
// each chunk's exact fp32 integers into int32 and sums them in registers.
//
// Every wait is bounded (globaltimer); a role that gives up records a
// timeout in the device status word, raises the CTA's abort flag, drains
// what it issued and returns, so the CTA always reaches its teardown and
// frees its tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace gp {

constexpr int kStatusTimeout = 4;  // GEMMPIPE_ERR_TIMEOUT

template <int BN_, int STAGES_, bool LDG_, bool INT_OUT_, bool CONVERT_ = false, int I8_STAGES_ = 1,
          bool PAIR_ = false, int CONV_GROUPS_ = 1, int CONV_WARPS_ = 4, bool TRACE_ = false, bool QUAD_ = false,
          int BK_ = 64>
struct GemmCfg {
    // TRACE: a copy of the kernel that stamps the pipelining trace (the
    // test hook gemmpipe_test_trace); the others carry no trace code.
    static constexpr bool TRACE = TRACE_;
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    // k values per stage: 64 (one 128-byte swizzle-atom row of fp16), or
    // 128 on CTA pairs: twice the bytes per copy and per barrier round trip.
    static constexpr int BK = BK_;
    // A stage holds A as BK / 64 sub-tiles of BM rows x 64 k (each in the
    // 128-byte swizzle) and B as 64-column atoms of BK rows.
    static constexpr int A_SUB_BYTES = BM * 128;
    static constexpr int B_ATOM_BYTES = BK * 128;
    static constexpr int STAGES = STAGES_;
    static constexpr bool LDG = LDG_;
    static constexpr bool INT_OUT = INT_OUT_;

    // PAIR: a cluster of two CTAs computes a 256 x BN tile with one
    // tcgen05.mma.cta_group::2 stream; each CTA holds 128 rows of A and
    // BN/2 columns of B, and receives its 128 rows of the accumulator.
    static constexpr bool PAIR = PAIR_;
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;
    static constexpr int CTA_BN = PAIR ? BN / 2 : BN;
    // QUAD: a cluster of two CTA pairs computes a 256 x 2BN tile, each pair
    // its own BN columns over the same 256 rows.  The pairs share A: each
    // CTA loads half of its 128 rows of a k-block and multicasts it to its
    // counterpart in the other pair, so an SM issues 24 KiB of copies per
    // k-block instead of 32 (copy issue per SM, not data arriving, is what
    // bounds the k-loop).
    static constexpr bool QUAD = QUAD_;
    static constexpr int CLUSTER = QUAD ? 4 : (PAIR ? 2 : 1);
    static constexpr int TILE_N = QUAD ? 2 * BN : BN;

    // Columns of one tcgen05.mma (N <= 256); a 512-wide pair tile issues
    // two per k-step into the two halves of one 512-column accumulator.
    // Each CTA of a pair holds, for every MMA, MMA_N / 2 columns of B.
    static constexpr int MMA_N = BN < 256 ? BN : 256;
    static constexpr int N_MMAS = BN / MMA_N;

    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BK * CTA_BN * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int NB64 = CTA_BN / 64;  // 64-column B atoms per stage
    static constexpr int NB64_PER_MMA = NB64 / N_MMAS;

    // CONVERT: int8 operands arrive by TMA in an int8 ring; converter warps
    // widen them to fp16 into the MMA's stage (INT8 path without a widening
    // pass); chunk partials are accumulated in C itself.
    static constexpr bool CONVERT = CONVERT_;
    static constexpr int I8_STAGES = CONVERT ? I8_STAGES_ : 0;
    static constexpr int I8_A_BYTES = BM * BK;
    static constexpr int I8_B_ATOMS = (PAIR_ ? BN_ / 2 : BN_) / 128;  // 128-column int8 atoms
    static constexpr int I8_B_BYTES = BK * 128 * I8_B_ATOMS;
    static constexpr int I8_STAGE_BYTES = I8_A_BYTES + I8_B_BYTES;

    static constexpr int PRODUCER_WARPS = LDG ? 8 : 1;
    static constexpr int PRODUCER_THREADS = 32 * PRODUCER_WARPS;
    static constexpr int CONV_WARPS = CONVERT ? CONV_WARPS_ : 0;
    static constexpr int CONV_THREADS = 32 * CONV_WARPS;
    static constexpr int CONV_GROUPS = CONV_GROUPS_;  // converter groups working on different k-blocks
    static_assert(CONV_WARPS == 0 || CONV_WARPS % CONV_GROUPS == 0, "groups of whole warps");
    static constexpr int MMA_WARP = PRODUCER_WARPS + CONV_WARPS;
    static constexpr int EPI_WARPS = 8;
    // Register split (TMA producer, no converter): warps 0-3 are the control
    // warpgroup (producer, MMA issuer, two idle warps) and hand registers to
    // the two epilogue warpgroups with setmaxnreg, so the INT8 epilogue
    // keeps its 128 running sums per thread in registers.  The shares add up
    // to the launch allocation of 384 threads x 168 registers.
    static constexpr bool REG_SPLIT = !LDG && !CONVERT;
    static constexpr int CTRL_REGS = 120;
    static constexpr int EPI_REGS = 192;
    static constexpr int EPI_WARP0 = REG_SPLIT ? 4 : MMA_WARP + 1;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int SPLIT_REGS = REG_SPLIT ? 32 * (4 * CTRL_REGS + EPI_WARPS * EPI_REGS) : 0;
    static_assert(!REG_SPLIT || (THREADS == 384 && SPLIT_REGS == THREADS * 168), "register split shares");
    // Running int32 sums of the INT8 chunks: in registers (128 per epilogue
    // thread) while the CTA has at most 12 warps -- 3 per scheduler, 168
    // registers each; with more warps they are kept in C itself.
    static constexpr bool SUM_IN_C = CONVERT && THREADS > 12 * 32;
    static constexpr int EPI_COLS = BN / 2;  // columns per epilogue warp
    // Two accumulators (tile t+1's MMAs run while tile t is stored), or
    // one of 512 columns for the 512-wide pair tile: TMEM holds 512.
    static constexpr int ACC_BUFS = BN == 512 ? 1 : 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;
    // The epilogue holds at most 128 accumulator values per thread at a
    // time: a 512-wide tile's 256 columns per warp go in two passes.
    static constexpr int EPI_PASS_COLS = EPI_COLS < 128 ? EPI_COLS : 128;
    static constexpr int EPI_PASSES = EPI_COLS / EPI_PASS_COLS;

    static constexpr int I8_OFF = STAGES * STAGE_BYTES;
    static constexpr int STAGING_OFF = I8_OFF + I8_STAGES * I8_STAGE_BYTES;
    static constexpr int STAGING_BYTES = EPI_WARPS * 32 * 128;
    static constexpr int CTL_OFF = STAGING_OFF + STAGING_BYTES;
    static constexpr int CTL_BYTES = 8 * (2 * STAGES + 2 * I8_STAGES + 5) + 16;
    static constexpr int SMEM_BYTES = 1024 + CTL_OFF + CTL_BYTES;  // + alignment slack

    static_assert(BN == 128 || BN == 256 || BN == 512, "BN must be 128, 256 or 512");
    static_assert(BN != 512 || (PAIR && !INT_OUT && !CONVERT),
                  "512-wide tiles: fp16 CTA pairs only (the INT8 epilogue keeps 128 int32 sums per thread)");
    static_assert(STAGES >= 1 && STAGES <= 16, "ring depth");
    static_assert(BK == 64 || (BK == 128 && !QUAD && !LDG && !CONVERT), "BK = 128: TMA producer, no quads");
    static_assert(!(LDG && INT_OUT), "INT8 operands are widened into an aligned workspace");
    static_assert(!CONVERT || (INT_OUT && !LDG && I8_STAGES >= 1), "converter variant is INT8 with TMA");
    static_assert(!PAIR || (BN >= 256 && !LDG), "pair variant: TMA producer, 256- or 512-wide tiles");
    static_assert(!QUAD || (PAIR && BN == 256 && !CONVERT), "quad variant: two CTA pairs of 256 x 256 tiles");
    static_assert(!CONVERT || I8_B_ATOMS >= 1, "int8 B atoms are 128 columns wide");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation is a power of two");
    static_assert(SMEM_BYTES <= 232448, "over the per-CTA shared-memory limit");
};

template <int STAGES, int I8_STAGES = 0>
struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t full_i8[I8_STAGES > 0 ? I8_STAGES : 1];
    uint64_t empty_i8[I8_STAGES > 0 ? I8_STAGES : 1];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded mbarrier wait.  False when the CTA is aborting or the wait ran out
// of time (then it records the timeout and raises the abort flag).
struct Waiter {
    volatile int *abort;
    int *status;
    uint64_t timeout_ns;

    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const
    {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((i & 15u) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort = 1;
                    atomicCAS(status, 0, kStatusTimeout);
                    return false;
                }
            }
        }
    }

    // Bounded wait until a global flag holds `epoch` (another unit's
    // partial sums are published).
    __device__ __forceinline__ bool wait_flag(const uint32_t *flag, uint32_t epoch) const
    {
        if (ld_acquire_u32(flag) == epoch) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            if (ld_acquire_u32(flag) == epoch) return true;
            __nanosleep(64);
            if ((i & 15u) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort = 1;
                    atomicCAS(status, 0, kStatusTimeout);
                    return false;
                }
            }
        }
    }

    // Used only while draining after an abort: ignores the abort flag.
    __device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) const
    {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity))
            if (globaltimer_ns() - t0 > limit_ns) return false;
        return true;
    }
};

constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

// One item of a unit's schedule: the k-blocks [kb0, kb1) of the output tile
// at (m0, n0).  kind 0: the whole tile; 1: a part of a split tile that ends
// before its last k-block (partial sums go to the unit's slot); 2: the part
// holding the last k-block (this unit adds the other parts and stores C).
struct Work {
    int64_t m0, n0;
    int64_t kb0, kb1;
    int64_t sk_tile;  // index among the split tiles
    int kind;
};

// Persistent schedule: unit = CTA (or CTA pair) index.
template <class Cfg>
__device__ __forceinline__ int64_t unit_index()
{
    return blockIdx.x / Cfg::CLUSTER;
}

// Start of a unit's range of split k-blocks (units[u] covers
// [sk_begin(u), sk_begin(u + 1)) of the tile-major split work).
__device__ __forceinline__ int64_t sk_begin(const GemmParams &p, int64_t unit)
{
    return p.sk_work * unit / p.units;
}

// A unit's items: its whole tiles (round-robin over units), then its split
// range from the last tile to the first.  The range's last item is the only
// one that can end inside a tile (kind 1), so it is published first; its
// first item, the only one that can hold a tile's last k-block after
// another unit's part (kind 2), comes last and waits only on lower units.
template <class Cfg>
struct WorkIter {
    int64_t dp, beg, pos;
    int64_t t;           // split tile of the next split item (they come last tile first)
    uint32_t per_group;  // tiles in a group of group_m tile rows

    __device__ __forceinline__ explicit WorkIter(const GemmParams &p)
    {
        const int64_t u = unit_index<Cfg>();
        dp = u;
        beg = sk_begin(p, u);
        pos = sk_begin(p, u + 1);
        t = pos > beg ? (pos - 1) / p.num_kb : 0;
        per_group = static_cast<uint32_t>(p.group_m) * static_cast<uint32_t>(p.tiles / p.m_tiles);
    }

    __device__ __forceinline__ bool next(const GemmParams &p, Work &w)
    {
        int64_t tile;
        if (dp < p.dp_tiles) {
            tile = dp;
            dp += p.units;
            w.kb0 = 0;
            w.kb1 = p.num_kb;
            w.kind = 0;
            w.sk_tile = -1;
        } else if (pos > beg) {
            const int64_t ts = t * p.num_kb;
            w.kb1 = pos - ts;
            w.kb0 = beg > ts ? beg - ts : 0;
            pos = ts + w.kb0;
            w.kind = w.kb1 < p.num_kb ? 1 : (w.kb0 > 0 ? 2 : 0);
            w.sk_tile = t;
            tile = p.dp_tiles + t;
            --t;
        } else {
            return false;
        }
        // Grouped order: tile -> (group, index in group); a group holds
        // gm tile rows (the last one may hold fewer) times all columns.
        // Tile indices fit 32 bits (2^31 tiles of C would not fit in device
        // memory), and 32-bit division is several times cheaper than 64-bit
        // on the producer's and epilogue's path.
        const uint32_t tl = static_cast<uint32_t>(tile);
        const uint32_t gmax = static_cast<uint32_t>(p.group_m), mt = static_cast<uint32_t>(p.m_tiles);
        const uint32_t g = tl / per_group, in = tl - g * per_group;
        const uint32_t first = g * gmax;
        const uint32_t gm = mt - first < gmax ? mt - first : gmax;
        const uint32_t col = in / gm;
        w.m0 = static_cast<int64_t>(first + (in - col * gm)) * Cfg::TILE_M;
        w.n0 = static_cast<int64_t>(col) * Cfg::TILE_N;
        return true;
    }
};

// ------------------------------------------------------------ TMA producer

template <class Cfg>
__device__ void producer_tma_i8(const GemmParams &p, const CUtensorMap *tA, const CUtensorMap *tB,
                                uint32_t sbase, Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w)
{
    // int8 tiles into this CTA's int8 ring: A box 64 (k) x 128 (rows), no
    // swizzle; B as atoms of 128 (n) x 64 (k) with the 128-byte swizzle.
    // In a CTA pair each CTA loads its own rows of A and half of B.
    const uint32_t rank = Cfg::PAIR ? cluster_ctarank() : 0u;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;
    int64_t kb_count = 0;
    bool ok = true;
    WorkIter<Cfg> it(p);
    Work wk;
    while (ok && it.next(p, wk)) {
        const int32_t m0 = static_cast<int32_t>(wk.m0 + rank * Cfg::BM);
        const int32_t n0 = static_cast<int32_t>(wk.n0 + rank * Cfg::CTA_BN);
        for (int64_t kb = wk.kb0; kb < wk.kb1; ++kb, ++kb_count) {
            if (!w.wait(smem_u32(&ctl->empty_i8[stage]), phase ^ 1u)) {
                ok = false;
                break;
            }
            if (!(blockIdx.x == 0 && kb_count == p.stall_kb)) {
                const uint32_t fb = smem_u32(&ctl->full_i8[stage]);
                const uint32_t sa = sbase + Cfg::I8_OFF + stage * Cfg::I8_STAGE_BYTES;
                const int32_t k0 = static_cast<int32_t>(kb * Cfg::BK);
                mbar_arrive_expect_tx(fb, Cfg::I8_STAGE_BYTES);
                tma_load_2d(sa, tA, fb, k0, m0);
#pragma unroll
                for (int a = 0; a < Cfg::I8_B_ATOMS; ++a)
                    tma_load_2d(sa + Cfg::I8_A_BYTES + a * 8192, tB, fb, n0 + 128 * a, k0);
                armed |= 1u << stage;
                armed_par = phase ? (armed_par | (1u << stage)) : (armed_par & ~(1u << stage));
            }
            if (++stage == Cfg::I8_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        for (int s = 0; s < Cfg::I8_STAGES; ++s)
            if (armed & (1u << s))
                w.wait_drain(smem_u32(&ctl->full_i8[s]), (armed_par >> s) & 1u, kDrainNs);
    }
}

// ------------------------------------------------------ int8 -> fp16 converters
//
// Four warps widen each int8 k-block into the fp16 stage the MMA reads.  A
// thread takes 16 int8 of one row (one 16-byte shared load), widens them
// (bias by 128, place under the fp16 exponent of 1024, subtract 1152: exact
// for every int8) and writes two 16-byte chunks in the 128-byte-swizzled
// layout.  The int8 rows are 64 (A) or BN (B) bytes long, so a warp's loads
// cover contiguous bytes; its stores hit each 16-byte bank group four times
// per 512 bytes, the minimum.

__device__ __forceinline__ void widen4_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
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

__device__ __forceinline__ void widen16_store(const uint4 &v, uint32_t dst_lo, uint32_t dst_hi)
{
    uint32_t o[8];
    widen4_f16(v.x, o[0], o[1]);
    widen4_f16(v.y, o[2], o[3]);
    widen4_f16(v.z, o[4], o[5]);
    widen4_f16(v.w, o[6], o[7]);
    st_shared_v4(dst_lo, o[0], o[1], o[2], o[3]);
    st_shared_v4(dst_hi, o[4], o[5], o[6], o[7]);
}

template <class Cfg>
__device__ void converter(const GemmParams &p, uint32_t sbase, Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl,
                          const Waiter &w)
{
    // CONV_GROUPS independent groups take alternate k-blocks (group g takes
    // the k-blocks whose running index is g modulo the group count), so
    // several k-blocks are widened at once and the latency of one group's
    // load / widen / store / fence / signal chain is hidden.
    constexpr int G = Cfg::CONV_GROUPS;
    constexpr int GT = Cfg::CONV_THREADS / G;  // threads per group
    const int ct = threadIdx.x - 32 * Cfg::PRODUCER_WARPS;
    const int g = ct / GT, gt = ct % GT;
    constexpr int A_PIECES = Cfg::BM * (Cfg::BK / 16);  // 16 int8 per piece
    constexpr int B_ROW_PIECES = Cfg::CTA_BN / 16;
    constexpr int B_PIECES = Cfg::BK * B_ROW_PIECES;
    constexpr int PIECES = A_PIECES + B_PIECES;
    static_assert(A_PIECES % GT == 0 && B_PIECES % GT == 0, "even split");
    constexpr int PER = PIECES / GT;  // pieces per thread per k-block
    constexpr int BATCH = (A_PIECES / GT) < 8 ? (A_PIECES / GT) : 8;
    static_assert((A_PIECES / GT) % BATCH == 0 && (B_PIECES / GT) % BATCH == 0, "batches do not straddle A and B");
    // In a CTA pair the fp16 stage is complete when both CTAs have signalled
    // the leader's full barrier.
    const bool to_leader = Cfg::PAIR;
    int64_t kcount = 0;
    WorkIter<Cfg> it(p);
    Work wk;
    while (it.next(p, wk)) {
        for (int64_t kb = wk.kb0; kb < wk.kb1; ++kb, ++kcount) {
            if (kcount % G != g) continue;
            const int si = static_cast<int>(kcount % Cfg::I8_STAGES);
            const uint32_t phi = static_cast<uint32_t>((kcount / Cfg::I8_STAGES) & 1);
            const int sf = static_cast<int>(kcount % Cfg::STAGES);
            const uint32_t phf = static_cast<uint32_t>((kcount / Cfg::STAGES) & 1);
            bool got = w.wait(smem_u32(&ctl->full_i8[si]), phi);
            got = got && w.wait(smem_u32(&ctl->empty[sf]), phf ^ 1u);
            if (!__all_sync(0xffffffffu, got)) return;
            const uint32_t ia = sbase + Cfg::I8_OFF + si * Cfg::I8_STAGE_BYTES;
            const uint32_t ib = ia + Cfg::I8_A_BYTES;
            const uint32_t fa = sbase + sf * Cfg::STAGE_BYTES;
            const uint32_t fb = fa + Cfg::A_BYTES;
#pragma unroll 1
            for (int b0 = 0; b0 < PER; b0 += BATCH) {
                // Shared loads of the batch first (they pipeline), then the
                // widening and the stores.
                uint4 v[BATCH];
                const bool isA = b0 < A_PIECES / GT;
#pragma unroll
                for (int i = 0; i < BATCH; ++i) {
                    if (isA) {
                        const int pc = gt + (b0 + i) * GT;
                        v[i] = ld_shared_v4(ia + (pc >> 2) * 64 + (pc & 3) * 16);
                    } else {
                        // B pieces run k-row fastest: eight lanes take eight
                        // consecutive k rows of one 16-column piece, which the
                        // 128-byte swizzle (int8 atoms on load, fp16 atoms on
                        // store) spreads over all banks.
                        const int pc = gt + (b0 + i - A_PIECES / GT) * GT;
                        const int kk = pc % Cfg::BK, jn = pc / Cfg::BK;
                        v[i] = ld_shared_v4(ib + (jn >> 3) * 8192 + kk * 128 + (((jn & 7) ^ (kk & 7)) << 4));
                    }
                }
#pragma unroll
                for (int i = 0; i < BATCH; ++i) {
                    if (isA) {
                        const int pc = gt + (b0 + i) * GT;
                        const int r = pc >> 2, j = pc & 3;  // row, 16-k piece of the 64-k row
                        const uint32_t row = fa + r * 128;
                        widen16_store(v[i], row + (((2 * j) ^ (r & 7)) << 4), row + (((2 * j + 1) ^ (r & 7)) << 4));
                    } else {
                        const int pc = gt + (b0 + i - A_PIECES / GT) * GT;
                        const int kk = pc % Cfg::BK, jn = pc / Cfg::BK;  // k row, 16-n piece
                        const uint32_t row = fb + (jn >> 2) * 8192 + kk * 128;
                        const int c0 = (jn & 3) * 2;
                        widen16_store(v[i], row + ((c0 ^ (kk & 7)) << 4), row + (((c0 + 1) ^ (kk & 7)) << 4));
                    }
                }
            }
            // Every store of the group reaches the async proxy, then one
            // thread signals the stage (and frees the int8 slot).
            fence_proxy_async_smem();
            named_barrier_sync(1 + g, GT);
            if (gt == 0) {
                if (to_leader)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->full[sf]), 0));
                else
                    mbar_arrive(smem_u32(&ctl->full[sf]));
                mbar_arrive(smem_u32(&ctl->empty_i8[si]));
            }
        }
    }
}

template <class Cfg>
__device__ void producer_tma(const GemmParams &p, const CUtensorMap *tA, const CUtensorMap *tB,
                             uint32_t sbase, Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w)
{
    // The whole producer warp runs the loop; one elected lane issues.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;  // per stage: armed at least once / parity of last arm
    int64_t kb_count = 0;
    bool ok = true;
    WorkIter<Cfg> it(p);
    Work wk;
    while (ok && it.next(p, wk)) {
        const int32_t m0 = static_cast<int32_t>(wk.m0);
        const int32_t n0 = static_cast<int32_t>(wk.n0);
        for (int64_t kb = wk.kb0; kb < wk.kb1; ++kb, ++kb_count) {
            if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->empty[stage]), phase ^ 1u))) {
                ok = false;
                break;
            }
            if (!(blockIdx.x == 0 && kb_count == p.stall_kb)) {
              if (elect_one_sync()) {
                const uint32_t fb = smem_u32(&ctl->full[stage]);
                const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
                const int32_t k0 = static_cast<int32_t>(kb * Cfg::BK);
                mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
#pragma unroll
                for (int a = 0; a < Cfg::BK / 64; ++a) tma_load_2d(sa + a * Cfg::A_SUB_BYTES, tA, fb, k0 + 64 * a, m0);
#pragma unroll
                for (int j = 0; j < Cfg::NB64; ++j)
                    tma_load_2d(sa + Cfg::A_BYTES + j * Cfg::B_ATOM_BYTES, tB, fb, n0 + 64 * j, k0);
                if constexpr (Cfg::TRACE) {
                    if (p.trace && blockIdx.x == 0 && kb_count < p.trace_n) p.trace[kb_count] = globaltimer_ns();
                }
              }
                __syncwarp();
                armed |= 1u << stage;
                armed_par = phase ? (armed_par | (1u << stage)) : (armed_par & ~(1u << stage));
            }
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        // Let every copy this warp started land before the CTA exits.
        for (int s = 0; s < Cfg::STAGES; ++s)
            if (armed & (1u << s))
                w.wait_drain(smem_u32(&ctl->full[s]), (armed_par >> s) & 1u, kDrainNs);
    }
}

// ------------------------------------------------- bounded-load producer
//
// The page's LDG-register variant, moved onto producer warps: each k-block's
// A and B tiles are read from global memory into registers with plain loads,
// then stored into the stage in the same swizzled layout TMA would write.
// Works for any 2-byte alignment of base and pitch: a row segment of 64 fp16
// (128 bytes) is fetched by 8 lanes as naturally aligned 16-byte words, each
// containing at least one byte of the row (so never outside the allocation),
// realigned across neighbouring lanes with shuffles and funnel shifts, and
// masked to zero outside the matrix (rows >= M or K, columns >= K or N).

struct SegLoad {
    uint4 lo, ex;
    uint32_t s;
    int nvalid;  // valid fp16 of this lane's 8 (0..8)
};

// Lane j of an 8-lane group, row segment starting at element e0 of a row of
// L valid elements (row_ok false: whole segment is zero).
__device__ __forceinline__ SegLoad seg_issue(const uint16_t *rowp, bool row_ok, int64_t e0, int64_t L, int j)
{
    SegLoad r;
    r.lo = make_uint4(0, 0, 0, 0);
    r.ex = make_uint4(0, 0, 0, 0);
    r.s = 0;
    r.nvalid = 0;
    if (row_ok) {
        const uintptr_t vlo = reinterpret_cast<uintptr_t>(rowp);
        const uintptr_t vhi = vlo + 2 * static_cast<uintptr_t>(L);
        const uintptr_t seg = vlo + 2 * static_cast<uintptr_t>(e0);
        r.s = static_cast<uint32_t>(seg & 15u);
        const uintptr_t base = seg - r.s;
        const uintptr_t a0 = base + 16 * static_cast<uintptr_t>(j);
        if (a0 < vhi && a0 + 16 > vlo) r.lo = ldg_nc_v4(reinterpret_cast<const void *>(a0));
        if (j == 7 && r.s != 0) {
            const uintptr_t a1 = base + 128;
            if (a1 < vhi && a1 + 16 > vlo) r.ex = ldg_nc_v4(reinterpret_cast<const void *>(a1));
        }
        const int64_t left = L - (e0 + 8 * j);
        r.nvalid = left <= 0 ? 0 : (left >= 8 ? 8 : static_cast<int>(left));
    }
    return r;
}

// All 32 lanes must call this (shuffles).  Stores the lane's 16 bytes.
__device__ __forceinline__ void seg_store(const SegLoad &r, int j, uint32_t dst)
{
    uint4 hi;
    hi.x = __shfl_down_sync(0xffffffffu, r.lo.x, 1, 8);
    hi.y = __shfl_down_sync(0xffffffffu, r.lo.y, 1, 8);
    hi.z = __shfl_down_sync(0xffffffffu, r.lo.z, 1, 8);
    hi.w = __shfl_down_sync(0xffffffffu, r.lo.w, 1, 8);
    if (j == 7) hi = r.ex;
    uint32_t o[4];
    realign16(r.lo, hi, r.s, o);
    if (r.nvalid < 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t keep = (2 * i < r.nvalid ? 0x0000FFFFu : 0u) | (2 * i + 1 < r.nvalid ? 0xFFFF0000u : 0u);
            o[i] &= keep;
        }
    }
    st_shared_v4(dst, o[0], o[1], o[2], o[3]);
}

template <class Cfg>
__device__ void producer_ldg(const GemmParams &p, uint32_t sbase, Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w)
{
    constexpr int GROUPS = Cfg::PRODUCER_THREADS / 8;  // row segments per pass
    constexpr int SEGS = Cfg::BM + Cfg::BK * Cfg::NB64;
    static_assert(SEGS % GROUPS == 0 && Cfg::BM % GROUPS == 0, "passes split evenly");
    constexpr int PASSES = SEGS / GROUPS;
    constexpr int BATCH = 4;
    static_assert(PASSES % BATCH == 0, "batches");

    const int tid = threadIdx.x;  // producers are threads 0 .. PRODUCER_THREADS-1
    const int j = tid & 7;
    const int gslot = tid >> 3;
    int stage = 0;
    uint32_t phase = 0;
    int64_t kb_count = 0;
    WorkIter<Cfg> it(p);
    Work wk;
    while (it.next(p, wk)) {
        const int64_t m0 = wk.m0;
        const int64_t n0 = wk.n0;
        for (int64_t kb = wk.kb0; kb < wk.kb1; ++kb, ++kb_count) {
            const int64_t k0 = kb * Cfg::BK;
            const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
            const uint32_t sb = sa + Cfg::A_BYTES;
            bool ok = true;
#pragma unroll 1
            for (int b0 = 0; b0 < PASSES; b0 += BATCH) {
                SegLoad ld[BATCH];
                uint32_t dst[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    const int sg = (b0 + u) * GROUPS + gslot;
                    if (sg < Cfg::BM) {
                        const int64_t row = m0 + sg;
                        const bool rv = row < p.M;
                        ld[u] = seg_issue(rv ? p.A + row * p.lda : p.A, rv, k0, p.K, j);
                        dst[u] = sa + sg * 128 + ((j ^ (sg & 7)) << 4);
                    } else {
                        const int gb = sg - Cfg::BM;
                        const int kk = gb / Cfg::NB64, jc = gb % Cfg::NB64;
                        const int64_t row = k0 + kk;
                        const bool rv = row < p.K;
                        ld[u] = seg_issue(rv ? p.B + row * p.ldb : p.B, rv, n0 + 64 * jc, p.N, j);
                        dst[u] = sb + jc * 8192 + kk * 128 + ((j ^ (kk & 7)) << 4);
                    }
                }
                if (b0 == 0) {
                    // The stage must be free before the first store into it.
                    const bool got = w.wait(smem_u32(&ctl->empty[stage]), phase ^ 1u);
                    ok = __all_sync(0xffffffffu, got);
                    if (!ok) break;
                }
#pragma unroll
                for (int u = 0; u < BATCH; ++u) seg_store(ld[u], j, dst[u]);
            }
            if (!ok) return;
            fence_proxy_async_smem();
            if (!(blockIdx.x == 0 && kb_count == p.stall_kb)) mbar_arrive(smem_u32(&ctl->full[stage]));
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------ pair (cta_group::2)
//
// Both CTAs of the pair run this producer.  Each loads its 128 rows of A and
// its half of the task's B columns into its own stage; every copy counts its
// bytes on the leader CTA's full[s], which the leader's producer arms with
// the bytes of both CTAs.  empty[s] of each CTA is released by the leader's
// multicast commit.
template <class Cfg>
__device__ void producer_tma_pair(const GemmParams &p, const CUtensorMap *tA, const CUtensorMap *tB,
                                  uint32_t sbase, Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w,
                                  uint32_t crank)
{
    // The whole producer warp runs the loop (its state and the copies'
    // coordinates stay warp-uniform); one elected lane issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;
    int64_t kb_count = 0;
    bool ok = true;
    constexpr uint32_t pair_bytes = 2u * Cfg::STAGE_BYTES;  // both CTAs' copies
    const uint32_t rank = crank & 1u;       // rank within the CTA pair
    const uint32_t pair_i = crank >> 1;     // pair within a quad
    const uint32_t leader = crank & ~1u;    // cluster rank of the pair's leader
    const bool stall_cta = blockIdx.x == 0 && p.stall_kb >= 0;
    const uint32_t full0 = smem_u32(&ctl->full[0]);
    const uint32_t full0_leader = mapa_shared(full0, leader);
    // Quads: this CTA's half of its A rows goes to it and to its counterpart
    // in the other pair (same rank within its pair).
    [[maybe_unused]] const uint16_t a_mask = static_cast<uint16_t>((1u << crank) | (1u << (crank ^ 2u)));
    WorkIter<Cfg> it(p);
    Work wk;
    while (ok && it.next(p, wk)) {
        const int32_t m0 = static_cast<int32_t>(wk.m0 + rank * Cfg::BM);
        // This CTA's share of B: for each MMA of the k-step, its half of
        // that MMA's MMA_N columns (a quad's second pair: the next BN).
        const int32_t n0 = static_cast<int32_t>(wk.n0 + pair_i * Cfg::BN + rank * (Cfg::MMA_N / 2));
        for (int64_t kb = wk.kb0; kb < wk.kb1; ++kb, ++kb_count) {
            if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->empty[stage]), phase ^ 1u))) {
                ok = false;
                break;
            }
            if (!(stall_cta && kb_count == p.stall_kb)) {
              if (elect_one_sync()) {
                const uint32_t fb_local = full0 + 8u * static_cast<uint32_t>(stage);
                const uint32_t fb = full0_leader + 8u * static_cast<uint32_t>(stage);  // the leader's full[s]
                const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
                const int32_t k0 = static_cast<int32_t>(kb * Cfg::BK);
                if (rank == 0) mbar_arrive_expect_tx(fb_local, pair_bytes);
                if constexpr (Cfg::QUAD) {
                    tma_load_2d_pair_mc(sa + pair_i * (Cfg::A_BYTES / 2), tA, fb, k0,
                                        m0 + static_cast<int32_t>(pair_i) * (Cfg::BM / 2), a_mask);
                } else {
#pragma unroll
                    for (int a = 0; a < Cfg::BK / 64; ++a) tma_load_2d_pair(sa + a * Cfg::A_SUB_BYTES, tA, fb, k0 + 64 * a, m0);
                }
                if (p.b_groups) {
                    // One 3-D copy per MMA: its NB64_PER_MMA 64-column groups,
                    // 8 KiB apart in shared memory as the 2-D copies place them.
#pragma unroll
                    for (int u = 0; u < Cfg::N_MMAS; ++u)
                        tma_load_3d_pair(sa + Cfg::A_BYTES + u * Cfg::NB64_PER_MMA * Cfg::B_ATOM_BYTES, tB, fb, 0, k0,
                                         (n0 + u * Cfg::MMA_N) / 64);
                } else {
#pragma unroll
                    for (int j = 0; j < Cfg::NB64; ++j)
                        tma_load_2d_pair(sa + Cfg::A_BYTES + j * Cfg::B_ATOM_BYTES, tB, fb,
                                         n0 + (j / Cfg::NB64_PER_MMA) * Cfg::MMA_N + 64 * (j % Cfg::NB64_PER_MMA),
                                         k0);
                }
                if constexpr (Cfg::TRACE) {
                    if (p.trace && blockIdx.x == 0 && kb_count < p.trace_n) p.trace[kb_count] = globaltimer_ns();
                }
              }
                __syncwarp();
                armed |= 1u << stage;
                armed_par = phase ? (armed_par | (1u << stage)) : (armed_par & ~(1u << stage));
            }
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (ok) {
        // The MMA commits of the last k-blocks arrive on this CTA's empty
        // barriers (the peer's from the leader's tensor cores): wait for
        // each stage's last phase so none is still in flight at exit.
        for (int s = 0; s < Cfg::STAGES && ok; ++s) {
            const uint32_t ph = s < stage ? phase ^ 1u : phase;  // phase of the stage's next use
            ok = __all_sync(0xffffffffu, w.wait(smem_u32(&ctl->empty[s]), ph ^ 1u));
        }
    }
    if (!ok) {
        if (rank == 0) {
            // The leader's full barriers count both CTAs' copies.
            for (int s = 0; s < Cfg::STAGES; ++s)
                if (armed & (1u << s))
                    w.wait_drain(smem_u32(&ctl->full[s]), (armed_par >> s) & 1u, kDrainNs);
        } else if (armed) {
            // The peer cannot observe its copies (they count on the leader's
            // barriers): give them a bounded time to land.
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 2000000ull) {
            }
        }
    }
}

// Leader CTA only (cluster rank `crank`, even): its MMA warp issues the
// pair's MMAs (one elected lane).  A stage is released to both CTAs of the pair -- and in a
// quad to the other pair too, whose A copies also land in these stages.
template <class Cfg>
__device__ void mma_issuer_pair(const GemmParams &p, uint32_t sbase, uint32_t tmem_base,
                                Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w, uint32_t crank, int lane)
{
    constexpr uint32_t idesc = umma_idesc_f16_f32(2 * Cfg::BM, Cfg::MMA_N, true);
    const uint16_t BOTH = static_cast<uint16_t>(3u << crank);              // this pair's two CTAs
    const uint16_t STAGE_MASK = Cfg::QUAD ? static_cast<uint16_t>(0xF) : BOTH;  // whoever writes the stages
    // Byte offset of the B columns of MMA u of a k-step within a stage's B.
    constexpr int B_MMA_BYTES = Cfg::NB64_PER_MMA * Cfg::B_ATOM_BYTES;
    // Per-stage, per-k-step descriptors are offsets of these two (see mma_issuer).
    const uint64_t dA0 = umma_desc_sw128(sbase, 16, 1024);
    const uint64_t dB0 = umma_desc_sw128(sbase + Cfg::A_BYTES, Cfg::B_ATOM_BYTES, 1024);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    bool issued = false, ok = true;
    [[maybe_unused]] int64_t nkb = 0;  // k-blocks seen ready (trace copies only)
    WorkIter<Cfg> it(p);
    Work wk;
    while (ok && it.next(p, wk)) {
        for (int64_t kc = wk.kb0; kc < wk.kb1 && ok; kc += p.kb_per_chunk) {
            const int64_t kend = kc + p.kb_per_chunk < wk.kb1 ? kc + p.kb_per_chunk : wk.kb1;
            if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d = tmem_base + acc * Cfg::BN;
            for (int64_t kb = kc; kb < kend; ++kb) {
                if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->full[stage]), phase))) {
                    ok = false;
                    break;
                }
                if constexpr (Cfg::TRACE) {
                    if (lane == 0 && p.trace && blockIdx.x == 0 && nkb < p.trace_n) {
                        p.trace[p.trace_n + nkb] = globaltimer_ns();
                        p.trace[2 * p.trace_n + nkb] = sm_clock64();
                    }
                    ++nkb;
                    __syncwarp();  // converged again for elect.sync
                }
                tc_fence_after_sync();
                const uint64_t so = static_cast<uint64_t>((stage * Cfg::STAGE_BYTES) >> 4);
                if (elect_one_sync()) {
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / 16; ++kk)
#pragma unroll
                        for (int u = 0; u < Cfg::N_MMAS; ++u)
                            umma_f16_pair(d + u * Cfg::MMA_N,
                                          dA0 + so + (((kk / 4) * Cfg::A_SUB_BYTES + (kk % 4) * 32) >> 4),
                                          dB0 + so + ((u * B_MMA_BYTES + kk * 2048) >> 4), idesc,
                                          (kb > kc || kk > 0) ? 1u : 0u);
                    umma_commit_pair(smem_u32(&ctl->empty[stage]), STAGE_MASK);
                }
                __syncwarp();
                issued = true;
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one_sync()) umma_commit_pair(smem_u32(&ctl->tfull[acc]), BOTH);
            __syncwarp();
            if constexpr (Cfg::ACC_BUFS == 2) {
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
    }
    if (ok) {
        // The accumulators' last releases -- including the peer's
        // epilogue arrivals on these barriers -- have landed before the
        // pair's final (relaxed) cluster barrier.  The parities are the
        // ones the next use of each buffer would wait for.
        ok = __all_sync(0xffffffffu, w.wait(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u));
        if constexpr (Cfg::ACC_BUFS == 2)
            ok = ok && __all_sync(0xffffffffu, w.wait(smem_u32(&ctl->tempty[acc ^ 1u]),
                                                      acc == 0 ? acc_phase ^ 1u : acc_phase));
    }
    if (!ok && issued) {
        if (elect_one_sync()) umma_commit_pair(smem_u32(&ctl->drain), static_cast<uint16_t>(1u << crank));
        __syncwarp();
        w.wait_drain(smem_u32(&ctl->drain), 0, kDrainNs);
    }
}

// ------------------------------------------------------------- MMA issuer

template <class Cfg>
__device__ void mma_issuer(const GemmParams &p, uint32_t sbase, uint32_t tmem_base,
                           Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w, int lane)
{
    constexpr uint32_t idesc = umma_idesc_f16_f32(Cfg::BM, Cfg::BN, true);
    // Stage s, k-step kk of the ring differ from stage 0, k-step 0 only in
    // the start-address field (address >> 4, bits [0,14)); shared memory
    // stays under 256 KB so the sum never carries out of that field.
    const uint64_t dA0 = umma_desc_sw128(sbase, 16, 1024);
    const uint64_t dB0 = umma_desc_sw128(sbase + Cfg::A_BYTES, Cfg::B_ATOM_BYTES, 1024);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    bool issued = false, ok = true;
    [[maybe_unused]] int64_t nkb = 0;  // k-blocks seen ready (trace copies only)
    WorkIter<Cfg> it(p);
    Work wk;
    while (ok && it.next(p, wk)) {
        for (int64_t kc = wk.kb0; kc < wk.kb1 && ok; kc += p.kb_per_chunk) {
            const int64_t kend = kc + p.kb_per_chunk < wk.kb1 ? kc + p.kb_per_chunk : wk.kb1;
            if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d = tmem_base + acc * Cfg::BN;
            for (int64_t kb = kc; kb < kend; ++kb) {
                if (!__all_sync(0xffffffffu, w.wait(smem_u32(&ctl->full[stage]), phase))) {
                    ok = false;
                    break;
                }
                if constexpr (Cfg::TRACE) {
                    if (lane == 0 && p.trace && blockIdx.x == 0 && nkb < p.trace_n) {
                        p.trace[p.trace_n + nkb] = globaltimer_ns();
                        p.trace[2 * p.trace_n + nkb] = sm_clock64();
                    }
                    ++nkb;
                    __syncwarp();  // converged again for elect.sync
                }
                tc_fence_after_sync();
                const uint64_t so = static_cast<uint64_t>((stage * Cfg::STAGE_BYTES) >> 4);
                if (elect_one_sync()) {
                    umma_f16(d, dA0 + so, dB0 + so, idesc, kb > kc ? 1u : 0u);
                    // k-step kk: A sub-tile kk / 4 (64 k each), 32 bytes per
                    // 16 k within it; B 16 rows of its atoms per 16 k.
#pragma unroll
                    for (int kk = 1; kk < Cfg::BK / 16; ++kk)
                        umma_f16(d, dA0 + so + (((kk / 4) * Cfg::A_SUB_BYTES + (kk % 4) * 32) >> 4),
                                 dB0 + so + (kk * 2048 >> 4), idesc, 1u);
                    umma_commit(smem_u32(&ctl->empty[stage]));
                }
                __syncwarp();
                issued = true;
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one_sync()) umma_commit(smem_u32(&ctl->tfull[acc]));
            __syncwarp();
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    if (!ok && issued) {
        // Every MMA this warp issued must finish before TMEM is freed.
        if (elect_one_sync()) umma_commit(smem_u32(&ctl->drain));
        __syncwarp();
        w.wait_drain(smem_u32(&ctl->drain), 0, kDrainNs);
    }
}

// --------------------------------------------------------------- epilogue

// Stores a 32 x 32 block of 32-bit results: lane l holds row row0 + l,
// columns col0 .. col0 + 31.  The block goes through the warp's staging tile
// (16-byte chunks XOR-swizzled by row, conflict-free both ways) so that each
// global store instruction writes whole 128-byte row pieces.
// TMA = false keeps the block on the load/store path even where C takes TMA
// stores (C that a later chunk reads back and adds to).
template <bool ADD = false, bool TMA = true>
__device__ __forceinline__ void store_block(const GemmParams &p, const CUtensorMap *tC, uint32_t stg,
                                            const uint32_t *r, int64_t row0, int64_t col0, int lane)
{
    if (row0 >= p.M || col0 >= p.N) return;  // warp-uniform
    if (!ADD && TMA && p.tma_store) {
        // The staging tile is in the 128-byte swizzle the C tensor map
        // declares; one TMA store writes the block (clipped at M and N).
        if (lane == 0) bulk_wait_read<0>();  // the previous block's store has read the tile
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            st_shared_v4(stg + lane * 128 + ((c ^ (lane & 7)) << 4), r[4 * c], r[4 * c + 1], r[4 * c + 2],
                         r[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tC, stg, static_cast<int32_t>(col0), static_cast<int32_t>(row0));
            bulk_commit();
        }
        return;
    }
    __syncwarp();  // every lane has read the previous block out of the staging tile
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(stg + lane * 128 + ((c ^ (lane & 7)) << 4), r[4 * c], r[4 * c + 1], r[4 * c + 2],
                     r[4 * c + 3]);
    __syncwarp();
    uint32_t *C = static_cast<uint32_t *>(p.C);
    if (ADD && p.vec_store) {
        // Read all eight 16-byte pieces of C first, then add and store, so
        // the reads are in flight together.
        uint4 old[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3), c = lane & 7;
            const int64_t grow = row0 + rr, gcol = col0 + 4 * c;
            old[it] = make_uint4(0, 0, 0, 0);
            if (grow < p.M && gcol + 4 <= p.N)
                old[it] = *reinterpret_cast<const uint4 *>(C + grow * p.ldc + gcol);
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3), c = lane & 7;
            const uint4 v = ld_shared_v4(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
            const int64_t grow = row0 + rr, gcol = col0 + 4 * c;
            if (grow < p.M && gcol < p.N) {
                uint32_t *dst = C + grow * p.ldc + gcol;
                if (gcol + 4 <= p.N) {
                    const uint4 o = old[it];
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
                } else {
                    dst[0] += v.x;
                    if (gcol + 1 < p.N) dst[1] += v.y;
                    if (gcol + 2 < p.N) dst[2] += v.z;
                }
            }
        }
    } else if (p.vec_store) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3), c = lane & 7;
            const uint4 v = ld_shared_v4(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
            const int64_t grow = row0 + rr, gcol = col0 + 4 * c;
            if (grow < p.M && gcol < p.N) {
                uint32_t *dst = C + grow * p.ldc + gcol;
                if (gcol + 4 <= p.N) {
                    if constexpr (ADD) {
                        const uint4 o = *reinterpret_cast<const uint4 *>(dst);
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
                    } else {
                        *reinterpret_cast<uint4 *>(dst) = v;
                    }
                } else {
                    dst[0] = ADD ? dst[0] + v.x : v.x;
                    if (gcol + 1 < p.N) dst[1] = ADD ? dst[1] + v.y : v.y;
                    if (gcol + 2 < p.N) dst[2] = ADD ? dst[2] + v.z : v.z;
                }
            }
        }
    } else {
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
            const uint32_t v = ld_shared_b32(stg + rr * 128 + ((((lane >> 2) ^ (rr & 7))) << 4) + ((lane & 3) << 2));
            const int64_t grow = row0 + rr, gcol = col0 + lane;
            if (grow < p.M && gcol < p.N) C[grow * p.ldc + gcol] = ADD ? C[grow * p.ldc + gcol] + v : v;
        }
    }
    __syncwarp();
}

// Partial-sum slots of split tiles: slot = CTA (2 * pair + rank for pairs),
// 128 x BN values as [epilogue warp][32-column block][32 x 32].  Within a
// block the 16-byte group i of lane l's row sits at uint4 index 32 i + l, so
// every access of a warp covers 512 contiguous bytes.
template <class Cfg>
__device__ __forceinline__ uint4 *part_block(const GemmParams &p, int64_t slot, int e, int jb)
{
    return reinterpret_cast<uint4 *>(p.partials + slot * (Cfg::BM * Cfg::BN) +
                                     (static_cast<int64_t>(e) * (Cfg::EPI_COLS / 32) + jb) * 1024);
}

template <class Cfg>
__device__ __forceinline__ int64_t slot_of(int64_t unit, uint32_t crank)
{
    return Cfg::CLUSTER * unit + crank;
}

__device__ __forceinline__ void write_part(uint4 *blk, const uint32_t *r, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) blk[32 * i + lane] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
}

template <bool INT>
__device__ __forceinline__ void add_part(const uint4 *blk, uint32_t *r, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = blk[32 * i + lane];
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (INT)
                r[4 * i + j] += x[j];
            else
                r[4 * i + j] = __float_as_uint(__uint_as_float(r[4 * i + j]) + __uint_as_float(x[j]));
        }
    }
}

// The lowest unit whose range holds k-blocks of split tile `sk_tile`.  The
// units from there up to this one's predecessor hold its earlier k-blocks
// (every range is non-empty: the split work has at least one k-block per
// unit).
template <class Cfg>
__device__ __forceinline__ int64_t first_part_unit(const GemmParams &p, int64_t sk_tile)
{
    const int64_t tile_start = sk_tile * p.num_kb;
    int64_t v = unit_index<Cfg>() - 1;
    while (v > 0 && sk_begin(p, v) > tile_start) --v;
    return v;
}

template <class Cfg>
__device__ void epilogue(const GemmParams &p, const CUtensorMap *tC, uint32_t sbase, uint32_t tmem_base,
                         Ctl<Cfg::STAGES, Cfg::I8_STAGES> *ctl, const Waiter &w, int warp, int lane, uint32_t crank)
{
    const uint32_t rank = crank & 1u;     // rank within the CTA pair
    const uint32_t pair_i = crank >> 1;   // pair within a quad
    const uint32_t leader = crank & ~1u;  // cluster rank of the pair's leader
    const int e = warp - Cfg::EPI_WARP0;  // 0..7
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int h = e >> 2;                  // column half of the tile
    constexpr int NCOLS = Cfg::EPI_COLS;   // this warp's columns
    constexpr int NB = NCOLS / 32;         // 32-column blocks
    constexpr bool INT = Cfg::INT_OUT;
    constexpr bool ISUM = INT && !Cfg::SUM_IN_C;  // int32 running sums in registers
    // HOLD (register-split variants, fp32 output): the warp copies its whole
    // accumulator slice into registers and frees the TMEM buffer before any
    // global traffic, so the MMA never waits on C stores or partial sums.
    // Otherwise it works one 32-column block at a time.
    constexpr bool HOLD = Cfg::REG_SPLIT && !INT;
    // A 512-wide tile gives each warp 256 columns: too many to hold.  It
    // copies them in passes of 128 and frees the accumulator after the last
    // pass's copy; the MMA of the next item waits for the earlier passes'
    // stores (this tile shape has no second accumulator to overlap with).
    constexpr bool HOLD_N = HOLD && Cfg::EPI_PASSES > 1;
    constexpr bool HOLD_1 = HOLD && !HOLD_N;
    constexpr int NBP = Cfg::EPI_PASS_COLS / 32;  // 32-column blocks per pass
    const uint32_t stg = sbase + Cfg::STAGING_OFF + e * (32 * 128);
    const int64_t me = unit_index<Cfg>();
    const int64_t my_slot = slot_of<Cfg>(me, crank);
    uint32_t acc = 0, acc_phase = 0;

    auto release = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            if constexpr (Cfg::PAIR)
                mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), leader));  // the leader's
            else
                mbar_arrive(smem_u32(&ctl->tempty[acc]));
        }
        if constexpr (Cfg::ACC_BUFS == 2) {
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        } else {
            acc_phase ^= 1u;
        }
    };
    // The other parts of a split tile must be published before they are
    // added.  Each is the first split item of a lower unit, which waits on
    // nothing to produce it.
    auto wait_parts = [&](int64_t v_lo) -> bool {
        bool got = true;
        for (int64_t v = me - 1; v >= v_lo && got; --v)
            got = w.wait_flag(&p.flags[slot_of<Cfg>(v, crank) * Cfg::EPI_WARPS + e], p.epoch);
        return __all_sync(0xffffffffu, got);
    };

    WorkIter<Cfg> it(p);
    Work wk;
    while (it.next(p, wk)) {
        const int64_t row0 = wk.m0 + rank * Cfg::BM + q * 32;
        const int64_t colb = wk.n0 + pair_i * Cfg::BN + h * NCOLS;
        const int64_t v_lo = wk.kind == 2 ? first_part_unit<Cfg>(p, wk.sk_tile) : me;
        if ((!HOLD || HOLD_N) && !ISUM && wk.kind == 2 && !wait_parts(v_lo)) return;
        // fp32 bits (HOLD) or int32 sums (ISUM)
        uint32_t val[(HOLD_1 || ISUM) ? NCOLS : (HOLD_N ? Cfg::EPI_PASS_COLS : 1)];
        if constexpr (ISUM) {
#pragma unroll
            for (int i = 0; i < NCOLS; ++i) val[i] = 0;
        }
        // fp32 output: one accumulation per item (the chunk is the whole
        // k-range); INT8: one per chunk of at most 1024 k values.
        for (int64_t kc = wk.kb0; kc < wk.kb1; kc += p.kb_per_chunk) {
            const bool got = w.wait(smem_u32(&ctl->tfull[acc]), acc_phase);
            if (!__all_sync(0xffffffffu, got)) return;
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * Cfg::BN + h * NCOLS;
            if constexpr (Cfg::SUM_IN_C) {
                // Whole tiles only.  Chunk partials are exact integers; the
                // first chunk stores them, later chunks add into C.  When a
                // later chunk will read C back, every chunk goes through the
                // load/store path, so its reads follow the earlier chunk's
                // writes in this warp's own program order (a TMA store
                // completes asynchronously); a single chunk may use TMA.
                const bool one_chunk = wk.kb1 - wk.kb0 <= p.kb_per_chunk;
#pragma unroll
                for (int jb = 0; jb < NB; ++jb) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + jb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
                    if (one_chunk)
                        store_block<false, true>(p, tC, stg, r, row0, colb + jb * 32, lane);
                    else if (kc == wk.kb0)
                        store_block<false, false>(p, tC, stg, r, row0, colb + jb * 32, lane);
                    else
                        store_block<true, false>(p, tC, stg, r, row0, colb + jb * 32, lane);
                }
            } else if constexpr (ISUM) {
                // Chunk partials are integers below 2^24 in magnitude: exact
                // in fp32, so the conversion is exact.
#pragma unroll
                for (int jb = 0; jb < NB; ++jb) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + jb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        val[jb * 32 + i] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
                }
            } else if constexpr (HOLD_1) {
#pragma unroll
                for (int jb = 0; jb < NB; ++jb)
                    tmem_ld_32x32b_x32(tbase + jb * 32, *reinterpret_cast<uint32_t(*)[32]>(&val[jb * 32]));
                tmem_wait_ld();
            } else if constexpr (HOLD_N) {
                // One accumulation per item (fp32 output).  The other parts
                // of a split tile were awaited at the start of the item.
#pragma unroll 1
                for (int ps = 0; ps < Cfg::EPI_PASSES; ++ps) {
#pragma unroll
                    for (int jb = 0; jb < NBP; ++jb)
                        tmem_ld_32x32b_x32(tbase + ps * Cfg::EPI_PASS_COLS + jb * 32,
                                           *reinterpret_cast<uint32_t(*)[32]>(&val[jb * 32]));
                    tmem_wait_ld();
                    if (ps == Cfg::EPI_PASSES - 1) release();
#pragma unroll
                    for (int jb = 0; jb < NBP; ++jb) {
                        const int b = ps * NBP + jb;
                        if (wk.kind == 1) {
                            write_part(part_block<Cfg>(p, my_slot, e, b), &val[jb * 32], lane);
                        } else {
                            for (int64_t v = me - 1; v >= v_lo; --v)
                                add_part<false>(part_block<Cfg>(p, slot_of<Cfg>(v, crank), e, b), &val[jb * 32], lane);
                            store_block(p, tC, stg, &val[jb * 32], row0, colb + b * 32, lane);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int jb = 0; jb < NB; ++jb) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + jb * 32, r);
                    tmem_wait_ld();
                    if (wk.kind == 1) {
                        write_part(part_block<Cfg>(p, my_slot, e, jb), r, lane);
                    } else {
                        for (int64_t v = me - 1; v >= v_lo; --v)
                            add_part<false>(part_block<Cfg>(p, slot_of<Cfg>(v, crank), e, jb), r, lane);
                        store_block(p, tC, stg, r, row0, colb + jb * 32, lane);
                    }
                }
            }
            if constexpr (!HOLD_N) release();
        }
        if constexpr (ISUM || HOLD_1) {
            // The accumulator is already free.  A split tile's other parts
            // are added in unit order (exact for integers; a fixed order for
            // fp32), then the slice goes to C or to this unit's slot.
            if (wk.kind == 2) {
                if (!wait_parts(v_lo)) return;
                for (int64_t v = me - 1; v >= v_lo; --v)
#pragma unroll
                    for (int jb = 0; jb < NB; ++jb)
                        add_part<INT>(part_block<Cfg>(p, slot_of<Cfg>(v, crank), e, jb), &val[jb * 32], lane);
            }
#pragma unroll
            for (int jb = 0; jb < NB; ++jb) {
                if (wk.kind == 1)
                    write_part(part_block<Cfg>(p, my_slot, e, jb), &val[jb * 32], lane);
                else
                    store_block(p, tC, stg, &val[jb * 32], row0, colb + jb * 32, lane);
            }
        }
        if (wk.kind == 1) {
            // Publish this warp's part: data first, then the flag.
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_u32(&p.flags[my_slot * Cfg::EPI_WARPS + e], p.epoch);
        }
    }
}

// ---------------------------------------------------------------- kernel

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_pipelined_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    auto *ctl = reinterpret_cast<Ctl<Cfg::STAGES, Cfg::I8_STAGES> *>(smem + Cfg::CTL_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]),
                      Cfg::LDG ? Cfg::PRODUCER_THREADS : (Cfg::CONVERT ? (Cfg::PAIR ? 2 : 1) : 1));
            // A quad's stages are written by both pairs' copies: released by both MMA threads.
            mbar_init(smem_u32(&ctl->empty[s]), Cfg::QUAD ? 2 : 1);
        }
        for (int s = 0; s < Cfg::I8_STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full_i8[s]), 1);
            mbar_init(smem_u32(&ctl->empty_i8[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tfull[b]), 1);
            mbar_init(smem_u32(&ctl->tempty[b]), (Cfg::PAIR ? 2 : 1) * Cfg::EPI_WARPS);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == Cfg::MMA_WARP) {
        if constexpr (Cfg::PAIR) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    if constexpr (!Cfg::LDG) {
        if (threadIdx.x == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (p.tma_store) tma_prefetch_desc(&tmC);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (Cfg::PAIR) cluster_sync();  // the leader's barriers exist before the peer signals them
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    // The set-up above touches no global memory, so it overlaps the end of
    // the previous grid on the stream; from here on its results are visible.
    pdl_wait();
    pdl_launch_dependents();
    const Waiter w{&ctl->abort, p.status, p.timeout_ns};
    const uint32_t rank = Cfg::PAIR ? cluster_ctarank() : 0u;  // rank in the cluster (pair, or quad)
    const bool pair_leader = (rank & 1u) == 0;
    if constexpr (Cfg::REG_SPLIT) {
        // Each role runs inside the branch that set its register share.
        if (warp < 4) {
            setmaxnreg_dec<Cfg::CTRL_REGS>();
            if (warp == 0) {
                if constexpr (Cfg::PAIR)
                    producer_tma_pair<Cfg>(p, &tmA, &tmB, sbase, ctl, w, rank);
                else
                    producer_tma<Cfg>(p, &tmA, &tmB, sbase, ctl, w);
                __syncwarp();
            } else if (warp == Cfg::MMA_WARP) {
                if constexpr (Cfg::PAIR) {
                    if (pair_leader) mma_issuer_pair<Cfg>(p, sbase, tmem_base, ctl, w, rank, lane);
                } else {
                    mma_issuer<Cfg>(p, sbase, tmem_base, ctl, w, lane);
                }
                __syncwarp();
            }
        } else {
            setmaxnreg_inc<Cfg::EPI_REGS>();
            epilogue<Cfg>(p, &tmC, sbase, tmem_base, ctl, w, warp, lane, rank);
            if (lane == 0) bulk_wait<0>();  // every C store issued by this warp has completed
            __syncwarp();
        }
    } else if (warp < Cfg::PRODUCER_WARPS) {
        if constexpr (Cfg::LDG) {
            producer_ldg<Cfg>(p, sbase, ctl, w);
        } else if constexpr (Cfg::CONVERT) {
            if (lane == 0) producer_tma_i8<Cfg>(p, &tmA, &tmB, sbase, ctl, w);  // single CTA or pair
        }
    } else if (warp < Cfg::MMA_WARP) {
        if constexpr (Cfg::CONVERT) converter<Cfg>(p, sbase, ctl, w);
    } else if (warp == Cfg::MMA_WARP) {
        if constexpr (Cfg::PAIR) {
            if (pair_leader) mma_issuer_pair<Cfg>(p, sbase, tmem_base, ctl, w, rank, lane);
        } else {
            mma_issuer<Cfg>(p, sbase, tmem_base, ctl, w, lane);
        }
        __syncwarp();
    } else {
        epilogue<Cfg>(p, &tmC, sbase, tmem_base, ctl, w, warp, lane, rank);
        if (lane == 0) bulk_wait<0>();  // every C store issued by this warp has completed
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (Cfg::PAIR) {
        // No peer still signals or reads this CTA after the barrier.  On
        // the normal path every cross-CTA arrival has already been observed
        // (the leader waited for the accumulators' last releases, the
        // producers for their stages' last MMA commits), so the barrier
        // needs no release ordering.  A CTA that aborted keeps it (a wait
        // that ran out in one CTA leaves its peer waiting on arrivals that
        // never come, so that one aborts too).
        const bool aborted = *reinterpret_cast<volatile int *>(&ctl->abort) != 0;
        if (!Cfg::REG_SPLIT || __syncthreads_or(aborted))
            cluster_sync();
        else
            cluster_sync_relaxed();
    }
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after_sync();
        if constexpr (Cfg::PAIR)
            tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gp
