// variants.h -- host-side table of the compiled kernel variants.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_params.h"
#include "gemmpipe.h"

namespace gp {

struct VariantInfo {
    int producer;  // 0 TMA, 1 bounded loads
    int int_out;   // 1: INT8 chunked integer epilogue
    int convert;   // 1: int8 tiles by TMA, widened to fp16 in shared memory
    int BM, BN, BK, stages;
    int i8_stages;
    int pair;  // 1: cluster of two CTAs, tcgen05.mma.cta_group::2, 256-row tiles;
               // 2: a quad (cluster of two such pairs sharing A), 256 x 2BN tiles
    int threads;
    int smem_bytes;
    int split_ok;  // 1: the epilogue can take split (stream-K) tiles
    int traced;    // 1: the copy that stamps the pipelining trace (test hook only)
};

using LaunchFn = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const GemmParams &,
                                 int grid, cudaStream_t);
using ClustersFn = int (*)();  // co-resident CTA pairs on the current device (pair variants)

struct Variant {
    VariantInfo info;
    LaunchFn launch;
    ClustersFn max_pairs;
};

// Each kernel translation unit exports its variants.
int variants_f16(const Variant **out);
int variants_s8(const Variant **out);

// Auxiliary kernels (aux_kernels.cu).
cudaError_t launch_widen_s8_f16(const int8_t *A, int64_t rowsA, int64_t colsA, uint16_t *A16, int64_t pitchA16,
                                const int8_t *B, int64_t rowsB, int64_t colsB, uint16_t *B16, int64_t pitchB16,
                                int sms, cudaStream_t s);
// Widens columns [0, cols) of a rows x cols int8 block with source pitch
// spitch into dst (pitch dpitch), writing only those columns (rounded up to
// 8 with zeros): a column slice of a wider matrix.
cudaError_t launch_widen_s8_f16_cols(const int8_t *src, int64_t rows, int64_t cols, int64_t spitch, uint16_t *dst,
                                     int64_t dpitch, int sms, cudaStream_t s);
cudaError_t launch_pad_f16(const uint16_t *src0, int64_t rows0, int64_t cols0, uint16_t *dst0, int64_t pitch0,
                           const uint16_t *src1, int64_t rows1, int64_t cols1, uint16_t *dst1, int64_t pitch1,
                           int sms, cudaStream_t s);
cudaError_t launch_zero_fill(void *dst, int64_t bytes, int sms, cudaStream_t s);
cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, int sms, cudaStream_t s);
cudaError_t status_word(int **ptr);  // device address of the current device's status word

// The legacy warp-MMA INT8 path (gemm_imma.cu): mma.sync m16n8k32 with a
// cp.async ring, on A and a transposed copy of B (comparison path).
bool imma_supported(const int8_t *A, int64_t K);
int64_t imma_bt_pitch(int64_t K);
cudaError_t launch_transpose_s8(const int8_t *B, int64_t K, int64_t N, int8_t *BT, int64_t ldbt, cudaStream_t s);
cudaError_t launch_imma_s8(const int8_t *A, const int8_t *BT, int64_t ldbt, int32_t *C, int64_t M, int64_t N,
                           int64_t K, int stages, cudaStream_t s);
void imma_plan_info(VariantInfo *f, int stages);  // stages: 2, else the default 4

// The INT8 flow with fixed, caller-provided scratch (gemmpipe_api.cpp), for
// the no-allocation entry point.
gemmpipe_status_t s8_check_fixed_scratch(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B,
                                         const int32_t *C, int64_t scratch_bytes);
gemmpipe_status_t s8_with_fixed_scratch(int64_t M, int64_t N, int64_t K, const int8_t *A, const int8_t *B,
                                        int32_t *C, cudaStream_t s, uint16_t *scratch, int64_t scratch_bytes);

}  // namespace gp
