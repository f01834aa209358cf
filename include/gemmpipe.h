/*
 * gemmpipe.h -- C ABI of libgemmpipe: the software-pipelined tiled GEMM
 * C = A * B on one NVIDIA GB300 (compute capability 10.3, sm_103a).
 *
 * The operation.  "Pipeline GPU Kernel" (skill page), opening summary and
 * Step 3: a tiled GEMM whose K loop is restructured so that the global loads
 * of K-tile n+1 overlap the tensor-core math on K-tile n.  The page works on
 * INT8 IGEMM (int32 accumulate) and FP16 HMMA GEMMs with A of shape M x K,
 * B of shape K x N and BM/BN/BK tiling.  Step 5 states that the pipelining
 * leaves the arithmetic unchanged, so each entry point's result is the plain
 * matrix product:
 *
 *     C[i][j] = sum over k < K of A[i][k] * B[k][j]
 *
 * Layout (every matrix): row-major and densely packed.
 *     A: M x K, element (i, k) at A[i*K + k]
 *     B: K x N, element (k, j) at B[k*N + j]
 *     C: M x N, element (i, j) at C[i*N + j]
 * C is overwritten (no alpha/beta: the pages define none).  A, B and C must
 * not overlap.  No alignment beyond the element size is required.  An fp16
 * operand whose base or row pitch is not a multiple of 16 bytes cannot be
 * read by the tensor-memory accelerator (TMA); gemm_f16f32 then copies it
 * into the library workspace with a padded, aligned pitch ("Pipeline GPU
 * Kernel", pitfalls list: pad the inputs, or fall back to bounds-checked
 * loads) and, where that workspace cannot be had or the bounded-load
 * producer is forced, reads it with bounds-checked loads instead.  Results
 * are the same either way.
 *
 * Ownership: the caller allocates A, B and C in device memory (cudaMalloc,
 * or managed memory) on the current device and keeps them alive until the
 * work on `stream` has finished.  The library keeps a device workspace per
 * (device, stream) for operand copies -- gemm_s8s8s32's operands widened to
 * fp16, and misaligned fp16 operands of gemm_f16f32 padded to aligned rows --
 * allocated with cudaMalloc on first need, grown when a larger problem needs
 * it (cudaFree then waits for the device), released by
 * gemmpipe_release_workspaces() or at unload.  A second workspace per
 * (device, stream) holds stream-K partial sums: when the output tiles leave
 * the persistent grid's last wave at most 4/5 full (or, with fewer tiles
 * than the grid holds, when spreading them cuts each CTA's k-blocks to a
 * third or less -- on single CTAs of a compute-bound GEMM, by 1536 k values
 * or more), the k-blocks of the last waves' tiles are split into equal
 * ranges over all CTAs and a split tile's parts
 * are added by the CTA holding its last k-block (128 x BN x 4 bytes per CTA
 * plus 64 KiB of flags; if it cannot be allocated, every tile runs whole
 * instead -- same result, no error).  gemm_f16f32 with 16-byte aligned operands and pitches
 * and a tile count that fills whole waves allocates nothing.
 *
 * Execution: every GEMM call is asynchronous on `stream` (a cudaStream_t;
 * NULL is the legacy default stream) and targets the current CUDA device.
 * A return of GEMMPIPE_OK means "validated and enqueued".  Errors found on
 * the device (a pipeline wait that ran out of time) are reported later by
 * gemmpipe_get_device_status().  No C++ exception crosses this interface.
 * Calls may come from several host threads; the library's own state is
 * guarded by a mutex.
 *
 * Error behaviour common to the GEMM entry points:
 *   - M, N or K negative, any of them above 2^31 - 1, a matrix of 2^56
 *     elements or more, a C of 2^31 or more 128 x 128 tiles
 *     (ceil(M/128) * ceil(N/128) > 2^31 - 1), a null A/B with
 *     M*N*K > 0, a null C with M*N > 0, a pointer not aligned to its element
 *     size, or a pointer the CUDA runtime does not know as device or managed
 *     memory                                   -> GEMMPIPE_ERR_INVALID_VALUE
 *   - M == 0 or N == 0                         -> GEMMPIPE_OK, nothing launched
 *   - K == 0 (the empty sum)                   -> C is set to zero
 *   - current device is not compute capability 10.3, or no CUDA device
 *                                              -> GEMMPIPE_ERR_UNSUPPORTED_DEVICE
 *   - a kernel launch is refused               -> GEMMPIPE_ERR_LAUNCH
 *   - workspace allocation fails               -> GEMMPIPE_ERR_OUT_OF_MEMORY
 */
#ifndef GEMMPIPE_H
#define GEMMPIPE_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMMPIPE_API __attribute__((visibility("default")))
#else
#define GEMMPIPE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *gemmpipe_stream_t;

/* IEEE 754 binary16 value stored as its 16-bit pattern (same bits as __half). */
typedef uint16_t gemmpipe_half_t;

typedef enum {
    GEMMPIPE_OK = 0,
    GEMMPIPE_ERR_INVALID_VALUE = 1,
    GEMMPIPE_ERR_UNSUPPORTED_DEVICE = 2,
    GEMMPIPE_ERR_LAUNCH = 3,
    GEMMPIPE_ERR_TIMEOUT = 4,
    GEMMPIPE_ERR_INTERNAL = 5,
    GEMMPIPE_ERR_OUT_OF_MEMORY = 6
} gemmpipe_status_t;

/*
 * INT8 x INT8 -> INT32 GEMM, the pages' IGEMM ("Pipeline GPU Kernel", Step 2,
 * decision thresholds measured on an INT8 IGEMM at 4096^3; "Analyze Kernel
 * Bottleneck", Step 4, the IGEMM reference point).
 *
 * A: M x K int8, B: K x N int8, C: M x N int32; exact integer result.
 * Entries whose exact value does not fit int32 wrap modulo 2^32 (for int8
 * operands that needs K > 131071).
 *
 * sm_103a has no integer tcgen05 MMA, so the operands are widened to fp16
 * (every int8 value is exact in fp16) and multiplied on the fp16 tensor-core
 * path with fp32 accumulation in chunks of at most 1024 k values.  Each
 * chunk's partial sums are integers of magnitude <= 2^24, exact in fp32;
 * they are converted to int32 and added.  The operands are first widened
 * into the library workspace, 2*(M*Kp + K*Np) bytes with Kp, Np = K, N
 * rounded up to a multiple of 8; calls on one stream share that stream's
 * workspace and are ordered by it.  With the plan override producer = 0 and
 * A, B on 16-byte boundaries with K and N multiples of 16, the kernel
 * instead loads int8 tiles and widens them in shared memory (no operand
 * copy; in single-CTA variants C also holds the running int32 sums between
 * chunks).
 */
GEMMPIPE_API gemmpipe_status_t gemm_s8s8s32(int64_t M, int64_t N, int64_t K,
                               const int8_t *A, const int8_t *B, int32_t *C,
                               gemmpipe_stream_t stream);

/*
 * FP16 x FP16 -> FP32 GEMM, the pages' HMMA GEMM ("Analyze Kernel
 * Bottleneck", Step 2 peak table, FP16 tensor core; "Pipeline GPU Kernel",
 * Step 5 tolerances for FP16 tensor-core results).
 *
 * A: M x K binary16, B: K x N binary16, C: M x N binary32.  Products are
 * accumulated in fp32 on the tensor cores; the summation order differs from
 * a sequential sum, so results agree with an fp64 reference to within fp32
 * accumulation error.  Allocates only the stream-K workspace described
 * above (and a padded copy of a misaligned operand).
 */
GEMMPIPE_API gemmpipe_status_t gemm_f16f32(int64_t M, int64_t N, int64_t K,
                              const gemmpipe_half_t *A, const gemmpipe_half_t *B,
                              float *C, gemmpipe_stream_t stream);

/*
 * gemm_s8s8s32 for callers that cannot let a library allocate GPU memory.
 * The pages have no counterpart of this entry point.
 *
 * Who needs it: a process that has planned every byte of device memory up
 * front (for example a server whose own pool owns all free memory, or code
 * with a certified static memory budget), and code on a latency-critical
 * path where a cudaMalloc or cudaFree inside the call would stall the whole
 * device.  gemm_s8s8s32 itself may cudaMalloc (and cudaFree) its workspace;
 * this entry point never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *
 * How: the fp16 copies of A and B live in one fixed scratch array of
 * GEMMPIPE_NOALLOC_SCRATCH_BYTES that the library declares statically in
 * device memory.  The CUDA runtime creates that array on a device when it
 * loads the library's device code there -- with lazy module loading (the
 * default), during the first call of this entry point on that device -- and
 * the device holds it until the process exits.  So make one call per device
 * at start-up, while memory is still free; a device without room for the
 * array gives GEMMPIPE_ERR_OUT_OF_MEMORY on that call.  The caller still
 * passes A, B and C.
 *
 * Limits and behaviour:
 *   - needs 2 * (M * Kp + K * Np) <= GEMMPIPE_NOALLOC_SCRATCH_BYTES, with
 *     Kp and Np = K and N rounded up to a multiple of 8 (e.g. M = N = K =
 *     2048 fits, 4096^3 does not); larger problems return
 *     GEMMPIPE_ERR_INVALID_VALUE before anything is launched;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and keeps it; make
 *     that first call before any stream capture, and do not reset the
 *     device (cudaDeviceReset) while the library is in use, since the kept
 *     address would then be stale;
 *   - all calls share the one array and it keeps whatever the last call
 *     left there; nothing in it has to start at zero, because each call
 *     writes every scratch element it later reads;
 *   - calls whose work overlaps on the GPU (different streams, or several
 *     host threads without ordering) race on the array and give wrong
 *     results: order them, e.g. on one stream;
 *   - otherwise the same arguments, result and errors as gemm_s8s8s32.
 */
#define GEMMPIPE_NOALLOC_SCRATCH_BYTES (16u << 20)
GEMMPIPE_API gemmpipe_status_t gemm_s8s8s32_noalloc(int64_t M, int64_t N, int64_t K,
                                                    const int8_t *A, const int8_t *B, int32_t *C,
                                                    gemmpipe_stream_t stream);

/*
 * The two GEMMs above with A, B and C in host memory: the call copies the
 * operands to the GPU, computes C and copies it back, overlapping the three.
 * The pages' method (loads of the next tile overlap the math on this one)
 * applied one level up, between the host link and the GPU.
 *
 * Arguments, layout and result: as gemm_s8s8s32 / gemm_f16f32, except that
 * A, B and C are host pointers (any pointer cudaMemcpy accepts: pageable or
 * page-locked host memory, also managed or device memory).
 *
 * How: A is copied in row panels of gemmpipe_host_panel_rows(M) rows, on a
 * copy stream of the library's; panel p's GEMM runs on `stream` as soon as
 * its rows and B have arrived; its rows of C are copied back on a second
 * library stream while later panels compute.  The INT8 call widens B once
 * and each panel's rows of A as they arrive.  When B holds at least 4 MiB
 * and N is a multiple of 32, the first panel's rows go first and B follows
 * in two column halves; the first panel is computed half by half, so C
 * starts coming back after half of B.
 *
 * Ordering and completion: the copies start after all work enqueued on
 * `stream` before the call, and work enqueued on `stream` after the call
 * starts after C has been written.  With page-locked A, B and C (e.g.
 * cudaHostAlloc or cudaHostRegister) the call is asynchronous: synchronize
 * `stream` before reading C.  With pageable memory the CUDA runtime makes
 * the copies synchronous, so the call returns when C has been written (the
 * copies back still overlap the later panels' GEMMs).  The caller keeps A,
 * B and C allocated and A, B unchanged until then.  Host-buffer calls on
 * one stream must be issued from one host thread, or under the caller's own
 * lock: the side streams and events kept for that stream are shared, and two
 * calls enqueued at the same time can interleave their event records, so
 * that a copy back waits on the other call's event and reads C rows before
 * they are written.
 *
 * Memory: device buffers for A, B and C (M*K + K*N + M*N*4 bytes for INT8,
 * 2*M*K + 2*K*N + 4*M*N for FP16) in a per-(device, stream) workspace, plus
 * what the device-pointer call allocates; two library streams and a few
 * events per (device, stream).  gemmpipe_release_workspaces frees them.
 *
 * Errors: as the device-pointer calls (GEMMPIPE_ERR_OUT_OF_MEMORY when the
 * buffers do not fit); a failure after some copies were enqueued still
 * leaves `stream` ordered after them.
 */
GEMMPIPE_API gemmpipe_status_t gemm_s8s8s32_host(int64_t M, int64_t N, int64_t K,
                                                 const int8_t *A, const int8_t *B, int32_t *C,
                                                 gemmpipe_stream_t stream);
GEMMPIPE_API gemmpipe_status_t gemm_f16f32_host(int64_t M, int64_t N, int64_t K,
                                                const gemmpipe_half_t *A, const gemmpipe_half_t *B,
                                                float *C, gemmpipe_stream_t stream);

/*
 * Rows per panel of the host-buffer calls: a quarter of M rounded up to a
 * multiple of 256, at least 512 (so M <= 512 is one panel, and there are at
 * most four).  Needs no
 * GPU.
 */
GEMMPIPE_API int64_t gemmpipe_host_panel_rows(int64_t M);

/*
 * Synchronizes `stream`, then reads and clears the current device's error
 * word.  Returns GEMMPIPE_ERR_TIMEOUT if a kernel of this library gave up on
 * a pipeline wait (every wait is bounded; the kernel then stops issuing
 * work, drains what it issued, frees its tensor memory and exits, leaving
 * the CUDA context usable; that call's C is undefined), GEMMPIPE_ERR_LAUNCH
 * if the CUDA runtime reports an error for the stream, else GEMMPIPE_OK.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_get_device_status(gemmpipe_stream_t stream);

/* Static, never-null English name of a status code. */
GEMMPIPE_API const char *gemmpipe_status_string(gemmpipe_status_t status);

/*
 * "Pipeline GPU Kernel", Step 2: the per-tile compute/load ratio
 *     2*BM*BN*BK / ((BM*BK + BK*BN) * elem_bytes)
 * (two flops per multiply-add over the bytes of one A tile and one B tile).
 * Returns a negative value if any argument is < 1.
 */
GEMMPIPE_API double gemmpipe_compute_load_ratio(int BM, int BN, int BK, int elem_bytes);

/*
 * "Pipeline GPU Kernel", Step 1, generalised from the page's double buffer to
 * an S-stage ring: stages * (BM*BK + BK*BN) * elem_bytes, the operand bytes
 * of the shared-memory ring (stages = 2 is the page's smem_doubled).
 * Returns -1 if any argument is < 1.
 */
GEMMPIPE_API int64_t gemmpipe_stage_smem_bytes(int BM, int BN, int BK, int elem_bytes, int stages);

/* Kernel plan chosen for one call; filled by gemmpipe_plan(). */
typedef struct {
    int producer;        /* 0: TMA producer warp, 1: bounded-load (LDG) producer warps,
                            2: warp-level integer MMA with a cp.async ring (comparison path) */
    int BM, BN, BK;      /* output tile (BM = 256 for a CTA pair) and k-block */
    int stages;          /* depth S of the shared-memory ring */
    int k_chunk;         /* k values accumulated in one TMEM accumulator before a drain */
    int threads;         /* threads per CTA */
    int cta_pair;        /* 1: clusters of two CTAs share one 256-row MMA (tcgen05 cta_group::2);
                            2: quads, two such pairs per cluster sharing A (BN is then the
                            quad's tile width, 512) */
    int grid;            /* persistent CTAs launched */
    int64_t tiles;       /* output tiles of BM x BN */
    int64_t units;       /* persistent units: CTAs, or CTA pairs */
    int64_t split_tiles; /* tiles whose k-blocks are split over units (stream-K; 0: every tile whole) */
    int64_t k_blocks;    /* ceil(K / BK) */
    int64_t smem_bytes;  /* dynamic shared memory per CTA */
    int vector_store;    /* 1: 16-byte stores of C, 0: 4-byte stores */
    int operand_copy;    /* 0: none (INT8: widened in the kernel), 1: int8 widened to fp16 in the
                            workspace, 2: misaligned fp16 padded in the workspace,
                            3: int8 B transposed in the workspace (producer 2) */
    int64_t workspace_bytes; /* library workspace the call needs (operand copies + split partial sums) */
} gemmpipe_plan_t;

/*
 * Fills *plan with the kernel configuration that gemm_s8s8s32 (dtype 0) or
 * gemm_f16f32 (dtype 1) would use for these arguments on the current device.
 * Launches nothing and dereferences no pointer.  A, B or C may be NULL: a
 * NULL pointer is planned as if it were 256-byte aligned.  Sizes are checked
 * as in the GEMM calls (INVALID_VALUE); M, N or K equal to 0 give an all-zero
 * plan.  Needs a compute capability 10.3 device (else UNSUPPORTED_DEVICE).
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_plan(int dtype, int64_t M, int64_t N, int64_t K,
                                const void *A, const void *B, const void *C,
                                gemmpipe_plan_t *plan);

/*
 * Overrides the plan for the following calls of this process (tests and the
 * stage/producer ablation).  producer: -1 automatic, 0 TMA (only honoured
 * where TMA can describe the operands; for gemm_s8s8s32 it selects the
 * in-kernel widening of int8 tiles), 1 bounded-load producer for
 * gemm_f16f32 and the workspace-widening path for gemm_s8s8s32, 2 (for
 * gemm_s8s8s32 with A on a 16-byte boundary and K a multiple of 16) the
 * pages' own design as a comparison path: warp-level integer MMA
 * (mma.sync m16n8k32) fed by a 4-stage cp.async ring, on A and a transposed
 * copy of B in the workspace (N x K bytes); exact like the other paths.  bn: 0
 * automatic, else 128, 256 or 512 (512: 256 x 512 tiles on CTA pairs, fp16
 * output only; where that variant does not apply, 256).  stages: 0 automatic, else one of the compiled
 * ring depths (when the chosen variant has no such depth the automatic one
 * is used; gemmpipe_plan reports what was taken).  cta_pair: -1 automatic,
 * 0 single CTAs, 1 CTA pairs where the shape allows them, 2 quads (a
 * cluster of two CTA pairs computing a 256 x 512 tile; each CTA loads half
 * of its rows of A and multicasts it to its counterpart in the other pair)
 * where the shape allows them.  split: -1
 * automatic, 0 every tile whole (no stream-K split), 1 split wherever the
 * schedule can (also where the automatic rule keeps whole tiles: a nearly
 * full last wave -- for quads one more than half full, or fewer than two
 * full waves --, a modest cut in k-blocks per CTA, memory-bound shapes
 * whose tiles already fill half the grid).  Returns INVALID_VALUE for values
 * outside these sets.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_set_plan_override(int producer, int bn, int stages, int cta_pair,
                                                          int split);

/*
 * Test hook: k values per pipeline stage for the following calls of this
 * process (0 automatic: 128 on fp16 single-CTA plans with N <= 128 unless
 * a ring depth is forced, 64 elsewhere; 64; or 128: 64 KiB stages, three
 * deep -- on CTA pairs, and on single CTAs with 128 x 128 fp16 tiles).  Plans without a 128-k variant
 * keep 64.  Returns INVALID_VALUE for other values.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_set_plan_bk(int bk);

/* Frees every workspace of the library (operand copies, stream-K partial
 * sums, host-call buffers) and the host calls' streams and events.  Call it
 * with no work of the library in flight. */
GEMMPIPE_API gemmpipe_status_t gemmpipe_release_workspaces(void);

/*
 * Kernel timing.  While enabled, every GEMM call records a CUDA event pair on
 * its stream around its main tensor-core kernel, and another around its
 * auxiliary kernels (INT8 widening, zero fill).  gemmpipe_timing_read waits
 * for the recorded events, returns the summed milliseconds and counts since
 * the previous read (any pointer may be NULL) and clears them.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_timing_enable(int enable);
GEMMPIPE_API gemmpipe_status_t gemmpipe_timing_read(double *gemm_ms, int64_t *gemm_launches,
                                       double *aux_ms, int64_t *aux_launches);

/* Total number of kernels this library has launched in this process. */
GEMMPIPE_API int64_t gemmpipe_launch_count(void);

/*
 * Device-to-device copy of `bytes` bytes by a plain streaming kernel (16-byte
 * accesses when both pointers and the size allow, else 1-byte).  It is the
 * in-run HBM bandwidth reference (blog page "Fixing a GPU kernel by hand --
 * making a transpose kernel 5x faster", section "Practice": a plain copy is
 * measured first as the upper bound of a memory-bound kernel).
 * Asynchronous on `stream`.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_copy(void *dst, const void *src, int64_t bytes,
                                gemmpipe_stream_t stream);

/*
 * Test hook for the bounded waits.  For the next GEMM launch only, CTA 0's
 * producer leaves its k-block number `k_block` (counted over the CTA's whole
 * schedule) unfilled, and every pipeline wait of that launch gives up after
 * `timeout_ms` milliseconds.  The consumer's wait therefore runs out; the
 * kernel records GEMMPIPE_ERR_TIMEOUT and exits cleanly.  k_block < 0 clears
 * the hook.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_test_inject_stall(int64_t k_block, int timeout_ms);

/*
 * Test hook that shows the pipelining ("Pipeline GPU Kernel", Steps 3-4:
 * the loads of the next K-tiles are issued while the tensor cores work on
 * this one).  For the next GEMM launch only, and when that launch runs the
 * FP16 CTA-pair kernel with 256-wide tiles and a 6- or 1-stage ring, with
 * 512-wide tiles, or on quads (the kernels compiled with the trace; any other
 * launch consumes the hook and records nothing),
 * CTA 0 (the leader CTA of pair 0) writes %globaltimer nanoseconds into `buffer`, a
 * device array of 3 * `entries` uint64: element j (j < entries) when its
 * producer has issued the tile copies of its j-th k-block (counted over the
 * CTA's whole schedule), element entries + j when its MMA thread finds that
 * k-block's data ready, just before issuing its MMAs, and element
 * 2 * entries + j the SM's %clock64 cycle count at that same moment (so
 * time per k-block can be split into cycles and clock rate).  Elements past
 * the CTA's k-blocks are left as they were.  entries = 0 clears the hook;
 * entries above 2^20, or a buffer that is not device memory, give
 * INVALID_VALUE.
 */
GEMMPIPE_API gemmpipe_status_t gemmpipe_test_trace(void *buffer, int64_t entries);

#ifdef __cplusplus
}
#endif

#endif /* GEMMPIPE_H */
