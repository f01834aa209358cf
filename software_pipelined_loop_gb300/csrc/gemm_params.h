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
    int64_t m_tiles, tiles;  // BM x BN tile grid (m fastest)
    int64_t full_tasks;      // tasks that are whole tiles: [0, full_tasks)
    int64_t tasks;           // whole tiles, then the tail tiles split into two BN/2 halves
    int64_t num_kb;        // ceil(K / BK)
    int64_t kb_per_chunk;  // k-blocks per TMEM accumulation unit
    int vec_store;         // C base and pitch allow 16-byte stores
    int64_t stall_kb;      // test hook: CTA 0 leaves this k-block unfilled (-1: none)
    uint64_t timeout_ns;   // bound of every pipeline wait
    int *status;           // device status word
};

}  // namespace gp
