/*
 * tcg.h -- C ABI of libtcg, a mixed-precision tensor-core GEMM for GB300
 * (sm_103a).
 *
 * The one operation (every entry point below serves it):
 *
 *     D = alpha * op(A) * op(B) + beta * C
 *
 *   - "Programming Tensor Cores in CUDA 9", section "什么是张量核?" and Figure 2:
 *     16-bit floating-point inputs, full-precision products, FP32 accumulation;
 *     C and D may be FP16 or FP32.
 *   - same page, section "如何在 cuBLAS 中使用张量核": the GemmEx argument list
 *     (transa, transb, m, n, k, alpha, A, Atype, lda, B, Btype, ldb, beta, C,
 *     Ctype, ldc, compute type); C is overwritten by D.  Its dimension rules
 *     (k, lda, ldb, ldc multiples of 8, m a multiple of 4) become the 16-byte
 *     rule below, and ragged m, n, k are supported.  Its silent fallback to a
 *     non-tensor-core routine is replaced by an explicit status.
 *   - same page, section "CUDA 9.0 中张量核的编程访问" (the wmma_example
 *     kernel): column-major storage with leading dimensions; alpha and beta
 *     applied elementwise to the accumulated product.
 *   - "CUDA Handbook, 17.5 Tensor Cores": TF32 mode, FP32 inputs rounded to
 *     TF32 (8-bit exponent, 10-bit mantissa) before the product, FP32
 *     accumulation.  libtcg rounds to nearest, ties to even.
 *   - "NVIDIA Tensor Core混合精度计算原理与应用解析", section 2.3: the final
 *     output is rounded to nearest even.
 *
 * Storage is column-major (BLAS).  op(A) is m x k, op(B) is k x n, C and D are
 * m x n and share the buffer C (D overwrites C; Ctype is both the C input type
 * and the D output type).  op(X) = X for TCG_OP_N and X^T for TCG_OP_T.  A
 * row-major problem D = A*B + C (A m x k, B k x n, all row-major) is the
 * column-major call gemm(N, N, n, m, k, alpha, B, n, A, k, beta, C, n).
 *
 * Supported (Atype = Btype, compute, Ctype) combinations; everything else
 * returns TCG_STATUS_NOT_SUPPORTED (no fallback of any kind):
 *     16F  / 32F            / 32F or 16F
 *     16BF / 32F            / 32F or 16BF
 *     32F  / 32F_FAST_TF32  / 32F
 *     32F  / 32F_3XTF32     / 32F
 *     8F_E4M3 or 8F_E5M2 (A and B alike) / 32F / 32F, 16F or 16BF
 *   FP8 inputs ("NVIDIA Tensor Core混合精度计算原理与应用解析", section 4.3.1: E4M3 and
 *   E5M2) are multiplied exactly and accumulated in FP32 like the 16-bit ones; their
 *   leading dimensions must be multiples of 16 elements (16 bytes).
 *
 * Ownership and threading.  The caller owns every device buffer; libtcg never
 * frees or keeps them.  The device-buffer calls accept only device memory of the
 * handle's device (cudaMalloc, stream-ordered pool or VMM allocations) for A, B, C
 * and the workspace: each pointer is checked with cudaPointerGetAttributes (once per
 * pointer value and handle; the last 16 that passed are remembered), and pageable,
 * pinned (cudaHostAlloc), managed or another device's memory is INVALID_VALUE with
 * nothing launched.  Host memory goes through the _host entry points.  All calls
 * are asynchronous on the handle's stream and return without a device
 * synchronisation (except tcg_get_device_error).  The GEMM kernel is launched with
 * programmatic stream serialization: it may be resident before the previous kernel
 * on the stream has finished, but it reads and writes no global memory until that
 * kernel has completed, so stream order is kept.  A handle is not thread-safe: use
 * one per host thread.  C must not overlap A or
 * B.  The first GEMM call on a handle binds it to the current device and
 * allocates a 4-byte device error word; make that call before any stream
 * capture.  The TF32 path and split-K calls need a workspace (see
 * tcg_set_workspace).  Once bound, and with its workspace large enough, a
 * handle's device-buffer calls can be captured in a CUDA graph: they then make
 * no allocation and no synchronisation (a pointer not seen before is checked in
 * relaxed capture mode), and replays give the eager results bit for bit.
 *
 * Pointers are device pointers (device memory of the handle's device, as above)
 * unless stated otherwise.
 */
#ifndef TCG_H_
#define TCG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TCG_STATUS_SUCCESS = 0,
    TCG_STATUS_NOT_INITIALIZED = 1,  /* no usable CUDA device / runtime */
    TCG_STATUS_INVALID_VALUE = 2,    /* argument check failed; nothing launched */
    TCG_STATUS_NOT_SUPPORTED = 3,    /* type combination not offered */
    TCG_STATUS_ARCH_MISMATCH = 4,    /* device is not compute capability 10.3 */
    TCG_STATUS_EXECUTION_FAILED = 5, /* a launch or CUDA call failed */
    TCG_STATUS_TIMEOUT = 6,          /* a bounded device wait gave up (sticky word) */
    TCG_STATUS_ALLOC_FAILED = 7      /* workspace / error word allocation failed */
} tcgStatus_t;

typedef enum { TCG_OP_N = 0, TCG_OP_T = 1 } tcgOp_t;

typedef enum {
    TCG_R_16F = 0,     /* IEEE binary16 */
    TCG_R_16BF = 1,    /* bfloat16: upper 16 bits of an IEEE binary32 */
    TCG_R_32F = 2,     /* IEEE binary32 */
    TCG_R_8F_E4M3 = 3, /* FP8 1/4/3, bias 7, no Inf, max 448 (inputs only) */
    TCG_R_8F_E5M2 = 4  /* FP8 1/5/2, bias 15, IEEE-style Inf/NaN (inputs only) */
} tcgDataType_t;

typedef enum {
    TCG_COMPUTE_32F = 0,            /* exact products, FP32 accumulation */
    TCG_COMPUTE_32F_FAST_TF32 = 1,  /* FP32 inputs rounded (RNE) to TF32 first */
    /* FP32 inputs as two TF32 words each, x = hi + lo with hi = RNE_tf32(x) and
     * lo = RNE_tf32(x - hi); D = alpha*(lo_A*hi_B + hi_A*lo_B + hi_A*hi_B) + beta*C,
     * three tensor-core products accumulated in FP32 (lo_A*lo_B, at most 2^-22 relative,
     * is dropped): multi-word emulation of a higher-precision product, "NVIDIA Tensor
     * Core混合精度计算原理与应用解析", section 5.1.  Accuracy against the exact product of
     * the FP32 inputs: |D - exact| <= (k + 8)*2^-23*(|alpha|*(|A||B|)_ij + |beta|*|C_ij|).
     * Needs twice the TF32 workspace. */
    TCG_COMPUTE_32F_3XTF32 = 2
} tcgComputeType_t;

typedef struct tcgContext *tcgHandle_t;

/* Create a handle.  Makes no CUDA call (device binding happens on first use).
 * Errors: INVALID_VALUE if h is NULL, ALLOC_FAILED if host memory runs out. */
tcgStatus_t tcg_create(tcgHandle_t *h);

/* Destroy a handle: synchronises its stream if it was used, frees the error
 * word and any workspace that libtcg allocated itself (never the caller's).
 * Errors: INVALID_VALUE if h is NULL. */
tcgStatus_t tcg_destroy(tcgHandle_t h);

/* Set the stream (a cudaStream_t passed as void*) for later calls; NULL is the
 * legacy default stream.  Errors: INVALID_VALUE if h is NULL. */
tcgStatus_t tcg_set_stream(tcgHandle_t h, void *stream);

/* Give the handle caller-owned device scratch memory for the TF32 path (which
 * writes TF32-rounded, K-major copies of op(A) and op(B) before the product) and for
 * the FP32 partial sums of split-K and tail-split calls (tcg_set_split_k).
 * ptr must be 256-byte aligned; bytes may be 0 to detach.  Without a caller
 * workspace the handle grows one of its own with cudaMalloc on the first TF32
 * call that needs more (not capture-safe).  Errors: INVALID_VALUE. */
tcgStatus_t tcg_set_workspace(tcgHandle_t h, void *ptr, size_t bytes);

/* Bytes of workspace a tcg_gemm_strided_batched call with these arguments
 * needs on the current device with the default kernel options: TF32 rounded copies,
 * plus the FP32 partial sums when the call splits K (see tcg_set_split_k) or cuts the
 * tiles of a partial last wave (tcg_tail_split_plan); 0 for an unsplit 16-bit or FP8
 * call.  Errors: INVALID_VALUE (NULL bytes). */
tcgStatus_t tcg_gemm_workspace_size(tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                                    int64_t k, tcgDataType_t Atype,
                                    tcgComputeType_t compute, int64_t batch_count,
                                    size_t *bytes);

/*
 * D = alpha*op(A)*op(B) + beta*C, column-major.
 *
 *   m, n, k      >= 0.  m == 0 or n == 0: no-op.  k == 0 or alpha == 0:
 *                D = beta*C and A, B are not read.  beta == 0: C is not read
 *                (NaN in C does not propagate).
 *   A, lda       op(A) data; lda >= m (OP_N) or >= k (OP_T), lda >= 1.
 *   B, ldb       op(B) data; ldb >= k (OP_N) or >= n (OP_T), ldb >= 1.
 *   C, ldc       in: C (read only if beta != 0); out: D.  ldc >= max(1, m).
 *   alpha, beta  FP32 scalars passed by value.
 *
 * Alignment (the TMA 16-byte rule): A, B, C 16-byte aligned; lda, ldb, ldc
 * times the element size a multiple of 16 bytes.
 *
 * Accuracy: FP32 accumulation of exact products; per element
 * |D - exact| <= k*2^-23*(|alpha|*(|A||B|)_ij + |beta|*|C_ij|), plus one output
 * ulp for 16-bit outputs (the error model of "NVIDIA Tensor Core混合精度计算原理
 * 与应用解析", section 2.3, with p = 23).  Integer-valued inputs whose sums stay
 * exact in FP32 give bit-exact results.
 *
 * Returns SUCCESS once the work is queued.  INVALID_VALUE: NULL handle or
 * needed pointer, negative sizes, ld too small, misaligned pointer or ld, a
 * pointer (or the caller's workspace) that is not device memory of the handle's
 * device.
 * NOT_SUPPORTED: type/compute combination.  ARCH_MISMATCH: not sm_103.
 * EXECUTION_FAILED: launch error, or the driver refused a tensor map (a leading
 * dimension or stride of 2^40 bytes or more; nothing launched).  ALLOC_FAILED:
 * first-use allocations.
 */
tcgStatus_t tcg_gemm_ex(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                        int64_t k, float alpha, const void *A, tcgDataType_t Atype,
                        int64_t lda, const void *B, tcgDataType_t Btype, int64_t ldb,
                        float beta, void *C, tcgDataType_t Ctype, int64_t ldc,
                        tcgComputeType_t compute);

/*
 * batch_count independent GEMMs; matrix i uses A + i*strideA, B + i*strideB,
 * C + i*strideC (strides in elements).  This is the strided-batched form of
 * tcg_gemm_ex, for many small problems in one launch ("NVIDIA Tensor Core混合
 * 精度计算原理与应用解析", section 6.2 item 3: merge small matrices into larger
 * units of work).  Same rules as tcg_gemm_ex, plus: batch_count >= 0 (0 is a
 * no-op); strides >= 0 and times the element size a multiple of 16 bytes;
 * strideC == 0 with batch_count > 1 is INVALID_VALUE (outputs would alias).
 */
tcgStatus_t tcg_gemm_strided_batched(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb,
                                     int64_t m, int64_t n, int64_t k, float alpha,
                                     const void *A, tcgDataType_t Atype, int64_t lda,
                                     int64_t strideA, const void *B, tcgDataType_t Btype,
                                     int64_t ldb, int64_t strideB, float beta, void *C,
                                     tcgDataType_t Ctype, int64_t ldc, int64_t strideC,
                                     int64_t batch_count, tcgComputeType_t compute);

/* The same two calls with A, B and C in HOST memory (pinned memory gives the full copy
 * bandwidth; pageable memory works).  The handle copies the operands into device buffers
 * it keeps (grown with cudaMalloc on demand, freed by tcg_destroy; not capture-safe), runs
 * the GEMM on its stream, copies D back into C and returns when C holds D.  The copies in
 * and out are pipelined against the product: column panels of B/C (tcg_gemm_ex_host) or
 * groups of batch entries (batched), up to four, each at least one wave of output tiles;
 * a single product of at least 8 waves goes as a grid of up to 4 x 4 blocks of D, each
 * block row of op(A) and block column of op(B) copied in once, in the order of first use.
 * Copies in run on one internal stream, copies out on another.  Arguments, layout rules
 * (leading dimensions and strides; no alignment needed for the host pointers), accuracy
 * and status codes as tcg_gemm_ex / tcg_gemm_strided_batched -- the result is theirs bit
 * for bit -- plus ALLOC_FAILED when the device buffers cannot be had.  Rows >= m inside
 * ldc and the gaps between batch entries of C are not written. */
tcgStatus_t tcg_gemm_ex_host(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                             int64_t k, float alpha, const void *A, tcgDataType_t Atype,
                             int64_t lda, const void *B, tcgDataType_t Btype, int64_t ldb,
                             float beta, void *C, tcgDataType_t Ctype, int64_t ldc,
                             tcgComputeType_t compute);
tcgStatus_t tcg_gemm_strided_batched_host(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb,
                                          int64_t m, int64_t n, int64_t k, float alpha,
                                          const void *A, tcgDataType_t Atype, int64_t lda,
                                          int64_t strideA, const void *B, tcgDataType_t Btype,
                                          int64_t ldb, int64_t strideB, float beta, void *C,
                                          tcgDataType_t Ctype, int64_t ldc, int64_t strideC,
                                          int64_t batch_count, tcgComputeType_t compute);

/*
 * TF32 GEMM that allocates nothing.  The pages have no counterpart to this entry
 * point: it exists for callers that cannot allocate device memory when they call
 * -- a latency-critical loop that cannot afford cudaMalloc/cudaFree (they
 * synchronise the device and take unbounded time), or a process whose device
 * memory belongs to another allocator (a framework's caching pool, a fixed
 * budget) that must not see raw allocations.
 *
 * Computes the same D = alpha*op(A)*op(B) + beta*C as tcg_gemm_ex with Atype =
 * Btype = Ctype = TCG_R_32F and TCG_COMPUTE_32F_FAST_TF32, with the same argument
 * rules and accuracy, on `stream` (a cudaStream_t; NULL = legacy default stream).
 * No handle: the caller passes inputs and outputs and nothing else.
 *
 * Scratch: the TF32-rounded operand copies live in one fixed 32 MiB device array
 * compiled into the library; every GPU that loads libtcg holds that array until
 * the process exits.  A call needs (m + n) * round_up(k, 4) * 4 bytes (each part
 * rounded up to 256 bytes) of it; larger problems return TCG_STATUS_NOT_SUPPORTED
 * before any device work (use tcg_gemm_ex with a workspace for them).
 *
 * All calls share that array, which keeps the last call's contents: calls that
 * overlap on the GPU (different streams, or different host threads without
 * ordering) race on it and give wrong results -- keep them on one stream or
 * otherwise ordered.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and the tensor-map encoder with that device current; make
 * that first call before any stream capture.  The addresses belong to the device's
 * context: after a cudaDeviceReset the next call finds a new context (by its id)
 * and looks them up again, so that first-call rule applies again too.  The call
 * makes no cudaMalloc, cudaFree or other allocating call.  A bounded device wait
 * that runs out stops the kernel early (output undefined) and sets a bit in a
 * device error word of these calls; tcg_noalloc_device_error reports it.
 *
 * Returns SUCCESS once queued; INVALID_VALUE for the argument errors of
 * tcg_gemm_ex (pointers are checked to be device memory of the current device on
 * every call: there is no handle to remember them in); NOT_SUPPORTED for problems beyond the scratch size;
 * ARCH_MISMATCH off sm_103; NOT_INITIALIZED / EXECUTION_FAILED for CUDA errors.
 */
tcgStatus_t tcg_gemm_tf32_noalloc(void *stream, tcgOp_t transa, tcgOp_t transb, int64_t m,
                                  int64_t n, int64_t k, float alpha, const float *A,
                                  int64_t lda, const float *B, int64_t ldb, float beta,
                                  float *C, int64_t ldc);

/* Status of the tcg_gemm_tf32_noalloc calls on the current device: synchronises
 * `stream` (a cudaStream_t; NULL = legacy default stream), then reads the calls'
 * device error word -- a sticky word in the library's own device memory that every
 * bounded wait that gave up since the last query has marked -- and clears it.
 * Returns SUCCESS, TIMEOUT (some call's kernel stopped early; its output is
 * undefined), or EXECUTION_FAILED if the synchronisation or the read failed;
 * NOT_INITIALIZED without a device.  Allocates nothing (plain symbol copies). */
tcgStatus_t tcg_noalloc_device_error(void *stream);

/* Synchronise the handle's stream, then return and clear the sticky device
 * error word: SUCCESS, or TIMEOUT if a bounded wait inside a kernel gave up
 * (the kernel then stopped early and its output is undefined), or
 * EXECUTION_FAILED if the synchronisation itself reported an error.  Returns
 * SUCCESS for a handle that has launched nothing.  INVALID_VALUE: NULL h. */
tcgStatus_t tcg_get_device_error(tcgHandle_t h);

/* Raw value of the last device error word read by tcg_get_device_error (bit
 * flags saying which wait gave up); 0 if none.  For diagnostics. */
uint32_t tcg_last_device_error_bits(tcgHandle_t h);

/* Static string naming a status. */
const char *tcg_status_string(tcgStatus_t s);

/* Test hooks.  wait_limit_ns bounds every device-side wait (0 restores the
 * default of 2 s).  fault_inject = 1 makes the next GEMM launches skip the
 * first operand load of the first tile, so the consumer's bounded wait runs
 * out and the kernel reports TIMEOUT through the error word (no fault, no
 * trap); 0 turns it off.  INVALID_VALUE: NULL h. */
tcgStatus_t tcg_set_debug(tcgHandle_t h, uint64_t wait_limit_ns, int fault_inject);

/* Clock probe, for measurement: the SM clock a GEMM kernel actually ran at.  on = 1
 * zeroes two device counters of the handle (allocated on first use) and makes every
 * later GEMM-kernel launch on h add, per CTA, the SM cycles (clock64) and the
 * nanoseconds (globaltimer) it ran for; on = 0 stops adding.  tcg_read_clock_probe
 * synchronises h's stream and returns the two sums: cycles / ns is the mean SM clock
 * in GHz over those launches (0 / 0 before any).  The kernels' other work is
 * unchanged.  INVALID_VALUE: NULL h or output pointer; ALLOC_FAILED,
 * EXECUTION_FAILED for CUDA errors. */
tcgStatus_t tcg_set_clock_probe(tcgHandle_t h, int on);
tcgStatus_t tcg_read_clock_probe(tcgHandle_t h, uint64_t *sm_cycles, uint64_t *ns);

/* Kernel options (0 = default for each).  cta_group: 2 (default) runs each 256x256
 * output tile on a pair of SMs (tcgen05 cta_group::2, B split between the pair's
 * shared memories); 1 runs 128x256 tiles on single SMs.  group_m: how many tile rows
 * the persistent scheduler walks together before moving along N (L2 reuse; default
 * 8).  Both variants meet the same accuracy bound.  INVALID_VALUE: NULL h,
 * cta_group outside 0..2, group_m outside 0..1024. */
tcgStatus_t tcg_set_kernel_options(tcgHandle_t h, int cta_group, int group_m);

/* Output tile width (not a step the pages describe -- a scheduling choice): 256
 * columns, or 128 for problems whose 256-wide tiles would fill at most half of the GPU's
 * SM pairs and that split K at neither width, so that a small problem's epilogue is
 * spread over twice the SMs (SM-pair kernel, FP16/BF16 inputs; other calls always use
 * 256).  tile_n: 0 (default) chooses so; 128 or 256 forces that width wherever a variant
 * exists.  Results are the same either way: every output element is accumulated in the
 * same K order (tcg_gemm_tile_plan reports the width a call uses).  INVALID_VALUE: NULL h,
 * other values. */
tcgStatus_t tcg_set_tile_n(tcgHandle_t h, int tile_n);

/* Where TCG_COMPUTE_32F_FAST_TF32 and TCG_COMPUTE_32F_3XTF32 calls round op(A) and op(B)
 * to TF32 (nearest even; the two-word split also writes x - hi, rounded, as a low word;
 * "CUDA Handbook, 17.5 Tensor Cores": FP32 inputs are rounded to TF32 on the way into the
 * tensor core).  Either way the rounded values land in the same K-major workspace copies
 * and the result is the same bit for bit; only the schedule differs:
 *   1  two pre-pass kernels round both operands, then the GEMM kernel reads the copies;
 *   2  the GEMM kernel rounds them itself: its epilogue warps, idle while an accumulator
 *      fills, round 64 x 128 blocks of the copies in the order the tiles need them, and
 *      the loads of a K range wait until its blocks are done, so the rounding's HBM
 *      traffic overlaps the multiplication instead of preceding it.  Slower for TF32 on
 *      GB300 (4096 x 4096 x 16384: 781 against 702 us per call): a tensor core fed at full
 *      rate leaves the SM's shared-memory/L1 data path too little room for the rounding.
 *   0  (default) 1 for TF32; for the two-word split (TCG_COMPUTE_32F_3XTF32, whose three
 *      products per stage leave the data path more room) 2 when K is not split and
 *      k >= 6144, else 1 (GB300: 4096 x 4096 x 16384 +4%, 2048 x 2048 x 8192 +3%,
 *      4096 x 4096 x 6144 +2%; k = 4096 even, shorter or split K lose).
 * In mode 2 the split's GEMM kernel writes both words.  Workspace: mode 2 needs a few
 * counters more (tcg_gemm_workspace_size includes them).
 * INVALID_VALUE: NULL h, other values. */
tcgStatus_t tcg_set_tf32_rounding(tcgHandle_t h, int mode);

/* K splitting ("split-K"; not a step the pages describe -- a scheduling choice of this
 * library for problems with few output tiles): the K range of every output tile is cut
 * into `splits` consecutive ranges, each range's products are accumulated on their own
 * (FP32, from zero), the partial sums land in an FP32 workspace and a second kernel adds
 * them in range order in FP32 before alpha, beta and the output rounding are applied.
 * The result stays inside the accuracy bound of tcg_gemm_ex; it is not the unsplit
 * accumulation bit for bit.
 * tcg_set_split_k: 0 (default) splits automatically -- only when the tiles (times the
 * batch) fill less than half of the GPU's SM pairs, into at most 64 ranges of at least
 * eight 128-byte K blocks each; 1 never splits; 2..64 forces that many ranges (fewer if
 * K is short).  INVALID_VALUE: NULL h, splits outside 0..64. */
tcgStatus_t tcg_set_split_k(tcgHandle_t h, int splits);

/* The split a problem of tiles output tiles (times batch) and num_k_blocks K blocks gets
 * on a GPU with `clusters` tile slots, with `forced` as in tcg_set_split_k: *splits
 * ranges (1: none) of *kb_per_split K blocks, the last one possibly shorter, none empty.
 * Pure host arithmetic, no device needed.  INVALID_VALUE: NULL outputs, negative
 * arguments, forced > 64. */
tcgStatus_t tcg_split_k_plan(int64_t tiles, int num_k_blocks, int clusters, int forced,
                             int *splits, int *kb_per_split);

/* Tail split (FP32 output, no split-K, automatic mode only): when the output tiles fill
 * whole waves of the GPU's SM pairs plus a partial one, the tiles of the partial wave
 * (or of it and the wave before) are cut into 2..4 K ranges whose FP32 partial sums
 * land in tile-sized workspace slices and are added in range order by a second kernel,
 * which then applies alpha and beta -- so the last wave takes a fraction of a tile's time.
 * Chosen when half the tensor time it is predicted to save (partial waves run at higher
 * clocks) exceeds the reduction's cost (a launch plus its memory traffic).
 * tcg_tail_split_plan is the rule, pure host arithmetic: tiles, K blocks (128 bytes of K
 * each), tile slots (clusters), one tile's time in microseconds, one tile's FP32 bytes
 * -> the number of whole tiles, the ranges (1: no tail split) and K blocks per range.
 * INVALID_VALUE: NULL outputs or negative counts. */
tcgStatus_t tcg_tail_split_plan(int64_t tiles, int num_k_blocks, int clusters, double tile_us,
                                double tile_bytes, int64_t *full_tiles, int *splits,
                                int *kb_per_split);

/* The K ranges of every output tile of the next call of this shape on h: *tile_m x *tile_n
 * tiles (column-major D), tile (b, mt, nt) at entry (b * tiles_m + mt) * tiles_n + nt of
 * splits[] (1: one accumulation over all of K) and k_per_split[] (K elements per range, the
 * last range possibly shorter).  max_tiles is the arrays' length (at least batch_count x
 * tiles_m x tiles_n).  Binds h to the current device.  INVALID_VALUE: NULL h or outputs,
 * negative sizes, unknown types, arrays too short. */
tcgStatus_t tcg_gemm_tile_plan(tcgHandle_t h, int64_t m, int64_t n, int64_t k,
                               tcgDataType_t Atype, tcgComputeType_t compute, tcgDataType_t Ctype,
                               int64_t batch_count, int64_t max_tiles, int *tile_m, int *tile_n,
                               int *splits, int64_t *k_per_split);

/* The split-K the next call of this shape on h will use (not the tail split; see
 * tcg_gemm_tile_plan): *splits ranges of *k_per_split K elements (the last one possibly
 * shorter).  Binds h to the current device like a GEMM call.  INVALID_VALUE: NULL h or outputs, negative sizes, unknown Atype. */
tcgStatus_t tcg_gemm_split_k(tcgHandle_t h, int64_t m, int64_t n, int64_t k,
                             tcgDataType_t Atype, tcgComputeType_t compute, int64_t batch_count,
                             int *splits, int64_t *k_per_split);

/* Number of GEMM-path kernel launches this handle has made (for the
 * benchmark's launch count).  Returns 0 for NULL. */
uint64_t tcg_launch_count(tcgHandle_t h);

#ifdef __cplusplus
}
#endif

#endif /* TCG_H_ */
