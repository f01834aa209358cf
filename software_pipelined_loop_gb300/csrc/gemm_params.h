// gemm_params.h -- kernel arguments of the pipelined GEMM, shared by host and
// device code.
#pragma once

#include <cstdint>

namespace gp {

struct GemmParams {
    int64_t M, N, K;
    const uint16_t *A;  // bounded-load producer only (TMA uses the tensor maps)
    int64_t lda;        // row pitch of A in elements
    const uint16_t *B;
    int64_t ldb;
    void *C;  // float or int32, M x N, row pitch ldc elements
    int64_t ldc;
    int64_t m_tiles, tiles;  // tile grid; a tile is 128 or 256 (CTA pair) rows x BN
    // Tile order: groups of group_m tile rows, m fastest inside a group and
    // the group's columns in turn, so the tiles in flight at once share a
    // few rows of A and columns of B (an L2-sized working set).
    int64_t group_m;
    // Persistent schedule over `units` (CTAs, or CTA pairs): tiles
    // [0, dp_tiles) go whole and round-robin; the k-blocks of the remaining
    // tiles (sk_work = their count times num_kb, tile-major) are split into
    // `units` equal contiguous ranges ("stream-K").  A unit whose range does
    // not start a tile leaves its partial sums in `partials` (one slot per
    // CTA) and publishes them with `epoch` in `flags`; the unit holding the
    // tile's first k-block adds them and stores C.
    int64_t units;
    int64_t dp_tiles;
    int64_t sk_work;
    uint32_t epoch;
    uint32_t *partials;  // fp32 or int32 values, 128 x BN per slot
    uint32_t *flags;     // one per (slot, epilogue warp)
    int64_t num_kb;        // ceil(K / BK)
    int64_t kb_per_chunk;  // k-blocks per TMEM accumulation unit
    int vec_store;         // C base and pitch allow 16-byte stores
    int tma_store;         // C blocks leave through TMA bulk-tensor stores (the C tensor map is valid)
    // B's tensor map is 3-D (64 columns x K rows x N / 64 column groups):
    // one copy brings a CTA's whole share of a B k-block (CTA pairs, N a
    // multiple of 64); otherwise 2-D, one copy per 64 columns.
    int b_groups = 0;
    int64_t stall_kb;      // test hook: CTA 0 leaves this k-block unfilled (-1: none)
    // Test hook: CTA 0 (the leader of pair 0) stamps %globaltimer into
    // trace[j] when its producer has issued the copies of its j-th k-block
    // and into trace[trace_n + j] when its MMA thread finds that k-block's
    // data ready, with the SM's %clock64 at that moment in
    // trace[2 * trace_n + j], for j < trace_n (nullptr: off).
    unsigned long long *trace = nullptr;
    int64_t trace_n = 0;
    uint64_t timeout_ns;   // bound of every pipeline wait
    int *status;           // device status word
};

}  // namespace gp
