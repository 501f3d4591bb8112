/*
 * dga.h -- dense GEMM on one GB300 (sm_103a): the C ABI.
 *
 * The one operation is the BLAS GEMM update
 *
 *     C <- alpha * A * B + beta * C,   A: M x K,  B: K x N,  C: M x N,
 *
 * as defined in "AI Programming: Matrix Product" (elainafan.one), section
 * "Dense matrix multiplication": alpha and beta let one call both scale the
 * product and accumulate into C.  Matrices are row-major, element (r, c) at
 * offset r*ld + c (same page, section "Row-major order"); B may instead be
 * column-major, which is how a Linear layer stores its weight (same page,
 * section "Fully-connected layer": Y = X * W^T with W of shape
 * [out_features, in_features]).
 *
 * Every call runs on the GPU, in kernels of this library; nothing falls back
 * to the CPU or to another library.  All calls are asynchronous on `stream`
 * and never synchronise, except dga_sync_status().
 *
 * Ownership: A, B, C and the workspace are caller-owned device memory (any
 * allocator, e.g. a PyTorch caching allocator).  The library allocates no
 * device memory and keeps no per-call state on the device beyond one status
 * word per kernel family.  C must not overlap A or B (detected, rejected).
 *
 * Thread safety: calls from several host threads are safe; dga_last_path()
 * and dga_last_cuda_error() are per host thread.
 */
#ifndef DGA_H_
#define DGA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* dga_stream_t;

/* Element types.  Supported (in, out) pairs:
 *   (DGA_F32, DGA_F32)    exact FP32 FFMA arithmetic, never TF32
 *   (DGA_BF16, DGA_F32)   bf16 inputs, fp32 accumulate, fp32 output
 *   (DGA_BF16, DGA_BF16)  bf16 inputs, fp32 accumulate, bf16 output (nearest-even)
 *   (DGA_F16, DGA_F32)    fp16 inputs, fp32 accumulate, fp32 output
 *   (DGA_F16, DGA_F16)    fp16 inputs, fp32 accumulate, fp16 output (nearest-even)
 *   (DGA_I8, DGA_I32)     int8 inputs, exact integer products and sums, int32
 *                         output; alpha*sum + beta*c is reduced mod 2^32.
 *   (DGA_TF32, DGA_F32)   opt-in, lossy: A and B are fp32 in memory, but the
 *                         tensor cores form each product from operands kept
 *                         to 10 fraction bits (TF32, "Matrix multiplication:
 *                         arithmetic intensity, tiling and Tensor Core",
 *                         sections 5.5 and 5.7), accumulating in fp32; each
 *                         product may be off by up to 2^-9 of its magnitude.
 *                         Never chosen for DGA_F32 inputs.  alpha, beta, C
 *                         and the bias are fp32 as for DGA_F32.            */
typedef enum { DGA_F32 = 0, DGA_BF16 = 1, DGA_F16 = 2, DGA_I8 = 3, DGA_I32 = 4, DGA_TF32 = 5 } dga_dtype;

/* Layout of B only; A and C are always row-major.
 *   DGA_ROW_MAJOR: B(k, j) = B[k*ldb + j], ldb >= max(1, N)
 *   DGA_COL_MAJOR: B(k, j) = B[j*ldb + k], ldb >= max(1, K)  (B stored N x K) */
typedef enum { DGA_ROW_MAJOR = 0, DGA_COL_MAJOR = 1 } dga_layout;

/* Kernel family.  DGA_PATH_AUTO picks the fastest one that accepts the
 * arguments; the others force one family (for tests and measurement) and make
 * the call fail with DGA_ERR_PATH when that family cannot run the arguments.
 *   GENERIC  any dtype pair, any layout, alignment or leading dimension
 *   SIMT     FP32 register-tiled FFMA kernel (F32 -> F32, K < 2^33)
 *   TCGEN05  5th-generation tensor cores, TMA + mbarrier pipeline, TMEM
 *            accumulators (BF16/F16 inputs, TF32 inputs; INT8 through exact
 *            bf16 encoding)
 *   SKINNY   bandwidth-bound kernel for M <= 16 with column-major B
 *            (decode-shaped X * W^T; BF16/F16 inputs)                          */
typedef enum {
    DGA_PATH_AUTO = 0,
    DGA_PATH_GENERIC = 1,
    DGA_PATH_SIMT = 2,
    DGA_PATH_TCGEN05 = 3,
    DGA_PATH_SKINNY = 4
} dga_path;

/* Status codes.  0 is success.  A negative value -p names the p-th argument
 * of dga_gemm_ex (1-based) as invalid, in the manner of BLAS's xerbla:
 *   -4 M < 0, -5 N < 0, -6 K < 0, -7 alpha NULL, -8 A NULL, -9 lda too small,
 *   -10 B NULL, -11 ldb too small, -12 beta NULL, -13 C NULL,
 *   -14 ldc too small, -15 workspace NULL while workspace_bytes > 0,
 *   -17 path not a dga_path value.                                          */
#define DGA_OK 0
#define DGA_ERR_UNSUPPORTED 1     /* (in, out) dtype pair or layout value not supported */
#define DGA_ERR_CUDA 2            /* a CUDA call failed; see dga_last_cuda_error()      */
#define DGA_ERR_DEVICE_TIMEOUT 3  /* a kernel gave up waiting (dga_sync_status only)    */
#define DGA_ERR_PATH 4            /* the forced path cannot run these arguments         */
#define DGA_ERR_WORKSPACE 5       /* workspace_bytes < dga_gemm_workspace_size(...)     */
#define DGA_ERR_OVERLAP 6         /* C overlaps A or B                                  */
#define DGA_ERR_DEVICE 7          /* current device is not sm_103 (GB300)               */
#define DGA_ERR_BAD_INDEX 8       /* a CSR index was out of range (dga_sync_status only) */

/*
 * dga_gemm -- C <- alpha*A*B + beta*C on `stream`, path chosen automatically.
 *
 *   in_dtype, out_dtype  one of the supported pairs above
 *   layout_b             DGA_ROW_MAJOR or DGA_COL_MAJOR (B only)
 *   M, N, K              sizes, >= 0
 *   alpha, beta          HOST pointers to the scalars: float for floating
 *                        point inputs (TF32 included), int32_t for DGA_I8 inputs.  beta == 0:
 *                        C is not read (NaN or Inf there does not propagate).
 *                        alpha == 0 or K == 0: A and B are not read.
 *   A, lda               device pointer, A(i, k) = A[i*lda + k], lda >= max(1, K)
 *   B, ldb               device pointer, see dga_layout
 *   C, ldc               device pointer, C(i, j) = C[i*ldc + j], ldc >= max(1, N)
 *   workspace            device scratch of at least workspace_bytes, or NULL
 *   workspace_bytes      bytes at `workspace`.  The tensor-core path needs
 *                        the bytes of its operand repacks (INT8 inputs; TF32
 *                        inputs with a row-major B; leading dimensions TMA
 *                        cannot express) and fails with DGA_ERR_WORKSPACE
 *                        without them.  dga_gemm_workspace_size() reports
 *                        those plus optional bytes: given them, the FP32 SIMT
 *                        path and, for floating point, the tensor-core CTA-pair
 *                        kernel split the tiles of a last, partly filled wave
 *                        along K (faster for tile counts that are not a
 *                        multiple of what runs at once; the parts are added in
 *                        a fixed order by a further launch, so results repeat
 *                        bit for bit); with less they run whole tiles.
 *   stream               CUDA stream the kernels are enqueued on
 *
 * M == 0 or N == 0 returns DGA_OK and touches no memory.  Returns a status
 * code; a kernel that timed out is reported later by dga_sync_status().
 */
int dga_gemm(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b,
             int64_t M, int64_t N, int64_t K,
             const void* alpha, const void* A, int64_t lda,
             const void* B, int64_t ldb, const void* beta,
             void* C, int64_t ldc,
             void* workspace, size_t workspace_bytes, dga_stream_t stream);

/*
 * dga_gemm_general -- the general form:
 *     C <- alpha * op(A) * op(B) + beta * C + bias
 * with the layout of A as well as of B, and an optional bias row, which is
 * the fully-connected layer of "AI Programming: Matrix Product", section
 * "Fully-connected layer" (Y = X W^T + b).
 *   layout_a   DGA_ROW_MAJOR: A(i, k) = A[i*lda + k], lda >= max(1, K)
 *              DGA_COL_MAJOR: A(i, k) = A[k*lda + i], lda >= max(1, M)
 *              (A stored K x M; e.g. the G^T of a weight gradient G^T X)
 *   bias       device pointer to N elements of the output type (int32_t for
 *              DGA_I8 inputs) added to every row of the result, or NULL.
 *              With alpha == 0 or K == 0 the result is beta*C + bias.
 * Argument errors are -(position in this list): -5 M, -6 N, -7 K, -8 alpha,
 * -9 A, -10 lda, -11 B, -12 ldb, -13 beta, -14 C, -15 ldc, -17 workspace,
 * -19 path; the bias must not overlap C (DGA_ERR_OVERLAP).  Other arguments
 * as for dga_gemm_ex.  The SKINNY family needs a row-major A; the tensor-core
 * family reads a column-major A in place (MN-major) and copies it into the
 * workspace only for INT8 (re-encoded as bf16 and transposed to K-major), for
 * TF32 (transposed to K-major) or when TMA cannot express lda (layout kept).
 */
int dga_gemm_general(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
                     dga_layout layout_b, int64_t M, int64_t N, int64_t K,
                     const void* alpha, const void* A, int64_t lda,
                     const void* B, int64_t ldb, const void* beta,
                     void* C, int64_t ldc, const void* bias,
                     void* workspace, size_t workspace_bytes, dga_path path,
                     dga_stream_t stream);

/* Workspace for dga_gemm_general, as dga_gemm_workspace_size is for dga_gemm_ex. */
size_t dga_gemm_general_workspace_size(dga_dtype in_dtype, dga_dtype out_dtype,
                                       dga_layout layout_a, dga_layout layout_b,
                                       int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t ldb, int64_t ldc, dga_path path);

/*
 * dga_sum_rows -- out[j] = sum over i < rows of G(i, j), j < cols, in fp32:
 * the bias gradient of the fully-connected layer (same page and section: the
 * output gradient summed over the batch).  G is row-major (G(i, j) =
 * G[i*ldg + j], ldg >= max(1, cols)) of DGA_F32, DGA_BF16 or DGA_F16; out is
 * a device array of cols floats.  The summation order is fixed, so results
 * are reproducible.  Errors: -2 rows < 0, -3 cols < 0, -4 G NULL, -5 ldg too
 * small, -6 out NULL; DGA_ERR_UNSUPPORTED for other dtypes.
 */
int dga_sum_rows(dga_dtype dtype, int64_t rows, int64_t cols, const void* G, int64_t ldg,
                 float* out, dga_stream_t stream);

/* dga_gemm with the kernel family forced (argument 17).  Same semantics. */
int dga_gemm_ex(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b,
                int64_t M, int64_t N, int64_t K,
                const void* alpha, const void* A, int64_t lda,
                const void* B, int64_t ldb, const void* beta,
                void* C, int64_t ldc,
                void* workspace, size_t workspace_bytes, dga_path path,
                dga_stream_t stream);

/* Bytes of workspace dga_gemm_ex can use for these arguments on `path`
 * (DGA_PATH_AUTO: the path dga_gemm would choose): required bytes for the
 * tensor-core path, optional bytes for the SIMT path (see dga_gemm).
 * Pointers are not needed: the answer depends on dtypes, layout, sizes,
 * leading dimensions and the current device's SM count (152 is assumed when
 * no device can be queried). */
size_t dga_gemm_workspace_size(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b,
                               int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc, dga_path path);

/* The path that dga_gemm_ex would run for these arguments (never AUTO), or a
 * negative status when the arguments are invalid.  A and B pointer alignment
 * matters: pass the real pointers. */
int dga_select_path(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b,
                    int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda, const void* B, int64_t ldb,
                    const void* C, int64_t ldc);

/* The dga_path of the last successful dga_gemm/dga_gemm_ex on this host thread
 * (DGA_PATH_AUTO if none yet or if the call did no GEMM work). */
int dga_last_path(void);

/* Number of kernels the last successful call on this host thread launched. */
int dga_last_launch_count(void);

/* Synchronises `stream`, then reads and clears the device status words the
 * kernels write when one of their bounded waits expires or (SpMV) when the
 * CSR arrays were malformed.  Returns DGA_OK, DGA_ERR_DEVICE_TIMEOUT,
 * DGA_ERR_BAD_INDEX, or DGA_ERR_CUDA when the synchronisation failed. */
int dga_sync_status(dga_stream_t stream);

/* Failure-detection self-test.  Enqueues one small kernel that waits on an
 * mbarrier nothing arrives at, using the same bounded wait as the GEMM
 * kernels, and gives up after limit_ns nanoseconds (0 < limit_ns <= 2e9,
 * else -1).  The next dga_sync_status(stream) must then report
 * DGA_ERR_DEVICE_TIMEOUT, and the GPU context stays usable.  Lets a caller
 * check the timeout path on its own GPU without faulting or hanging it.
 * The pages have no counterpart (their kernels have no waits). */
int dga_selftest_bounded_wait(int64_t limit_ns, dga_stream_t stream);

/*
 * Measurement helper, not part of any GEMM: a probe of the FP32 FMA rate.
 * The roofline of "Matrix multiplication: arithmetic intensity, tiling and
 * Tensor Core" (section 5.1) caps a compute-bound kernel at the chip's peak;
 * for the FP32 SIMT path that peak is derived as SMs x 128 lanes x 2 FLOP x
 * SM clock, and this probe measures what the FMA pipe sustains so the
 * derived figure can be checked.
 *
 * Enqueues one kernel on `stream`: 4 CTAs of 256 threads per SM, each thread
 * running 8 independent accumulator chains for `iters` iterations of 64
 * fused multiply-adds -- scalar fp32 FMAs (packed = 0) or fma.rn.f32x2 pairs
 * (packed = 1, the form the SIMT GEMM issues).  Time it with events around
 * the call; *flops (host pointer) receives the FLOPs the launch performs
 * (2 per FMA).  `out` is caller-owned device memory of at least
 * dga_probe_fp32_fma_out_floats() floats (one sum per thread, written so the
 * work cannot be dropped).
 * Errors: -1 packed not 0 or 1; -2 iters outside [1, 2^20]; -3 out null;
 * -4 out_floats too small; -5 flops null; DGA_ERR_DEVICE, DGA_ERR_CUDA.
 */
int dga_probe_fp32_fma(int packed, int64_t iters, float* out, int64_t out_floats, double* flops,
                       dga_stream_t stream);

/* Floats of `out` that dga_probe_fp32_fma writes on the current device
 * (152 SMs assumed when no device can be queried); also the int32 values
 * dga_probe_int8_mma writes. */
int64_t dga_probe_fp32_fma_out_floats(void);

/*
 * Measurement helper, not part of any GEMM: the rate of the integer tensor
 * instruction an exact INT8 GEMM could use instead of this library's bf16
 * encoding (mma.sync.m16n8k32 with s8 operands and s32 accumulators; the
 * tcgen05 integer kind is not available for sm_103a).  Enqueues one kernel:
 * 4 CTAs of 256 threads per SM, each warp running 8 independent accumulator
 * chains of `iters` steps on operands held in registers (the instruction's
 * best case).  Every lane of warp w holds A bytes c = w % 5 + 1 and B bytes
 * -2, so thread t writes out[t] = -2048 * c * iters, whatever the fragment
 * layout.  *ops (host pointer) receives the integer operations of the launch
 * (2 * 16 * 8 * 32 per instruction); time it with events around the call.
 * `out`: device memory of at least dga_probe_fp32_fma_out_floats() int32.
 * Errors: -1 iters outside [1, 2^17]; -2 out null; -3 out_ints too small;
 * -4 ops null; DGA_ERR_DEVICE, DGA_ERR_CUDA.
 */
int dga_probe_int8_mma(int64_t iters, int32_t* out, int64_t out_ints, double* ops,
                       dga_stream_t stream);

/*
 * Measurement helper, not part of any GEMM: the naive GEMM of "GEMM
 * optimisation, part 0" (chongfengling.github.io), section 2 -- one thread
 * per element of C, accumulating A(i, k) * B(k, j) over k in fp32 (fused
 * multiply-adds in ascending k), launched in blocks of 16 x 16 threads with
 * the block's x along the columns of C.  It is the kernel whose hardware
 * counters that page prints (section 2.3: at M = N = K = 2048, 536,870,912
 * global load requests and 1,073,741,824 sectors), kept so that the counter
 * method behind this library's profiles can be checked against them.
 *
 * C <- A * B with A (M x K), B (K x N) and C (M x N) row-major and contiguous
 * (leading dimensions K, N and N), device pointers, enqueued on `stream`.
 * Errors: -1 M, -2 N outside [1, 65536]; -3 K outside [1, 65536] or a matrix
 * of 2^31 elements or more; -4 A, -5 B, -6 C null; DGA_ERR_DEVICE,
 * DGA_ERR_CUDA.
 */
int dga_probe_naive_sgemm(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                          dga_stream_t stream);

/* The cudaError_t value behind the last DGA_ERR_CUDA on this host thread. */
int dga_last_cuda_error(void);

/* A static string naming a status code. */
const char* dga_status_string(int status);

/*
 * dga_gemm_i8_noalloc -- INT8 x INT8 -> INT32 GEMM that allocates nothing and
 * takes no workspace.  The pages have no counterpart: this entry point exists
 * for callers that cannot allocate device memory at all -- a plugin handed
 * only its input and output buffers, an engine that reserves all device
 * memory at start-up and forbids allocations afterwards, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.
 *
 * Same computation and argument meanings as dga_gemm with in_dtype = DGA_I8,
 * out_dtype = DGA_I32 (alpha, beta: host pointers to int32_t; A, B, C device
 * pointers; result alpha*A*B + beta*C reduced mod 2^32), run on the tensor
 * cores.  Instead of a caller workspace it uses one scratch area of
 * DGA_NOALLOC_SCRATCH_BYTES compiled into the library:
 *   - every GPU on which it is called holds that area until the process exits;
 *   - the call is refused with DGA_ERR_WORKSPACE, before anything is
 *     enqueued, when the operands re-encoded as bf16 exceed it: A takes
 *     M * round_up(K, 8) * 2 bytes and B N * round_up(K, 8) * 2 bytes in
 *     either layout (both are re-encoded K-major; each rounded up to 256
 *     bytes); e.g. M = 4093, N = 4099, K = 4096 (64 MiB) fits;
 *   - all calls share the area and it keeps the last call's contents
 *     (nothing in it needs to start at zero: each call rewrites all it reads);
 *     calls that overlap on the GPU -- other streams, other host threads --
 *     race on it, so serialise them;
 *   - the first call in a CUDA context (normally: the first call on each
 *     device, in its primary context) looks up the area's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is kept per context, so after cudaDeviceReset, or in another
 *     context on the same device, the next call looks it up again.
 * Argument errors are -(position in this function's argument list).  The
 * product always runs on the tensor-core path: where that path is
 * unavailable on the device (no tensor-map encoder in the driver, or not an
 * sm_103 GPU) the call returns DGA_ERR_PATH (or DGA_ERR_DEVICE) rather than
 * falling back to another kernel as dga_gemm does.  Other codes as for
 * dga_gemm_ex.
 */
#define DGA_NOALLOC_SCRATCH_BYTES (72ull << 20)
int dga_gemm_i8_noalloc(dga_layout layout_b, int64_t M, int64_t N, int64_t K,
                        const int32_t* alpha, const int8_t* A, int64_t lda,
                        const int8_t* B, int64_t ldb, const int32_t* beta,
                        int32_t* C, int64_t ldc, dga_stream_t stream);

/*
 * dga_spmv_csr -- y <- alpha * A * x + beta * y for a sparse rows x cols
 * matrix A in CSR form: the SpMV of "AI Programming: Matrix Product",
 * sections "CSR" and "SpMV".  Row i holds the entries p in the half-open
 * interval [row_offsets[i], row_offsets[i+1]), entry p being values[p] in
 * column column_indices[p]; y[i] gets the sum over those p of
 * values[p] * x[column_indices[p]] (fp32 products and sums, any order within
 * the tolerance 1e-4 * sum |a x| of the result; the order is fixed, so
 * results repeat bit for bit).  Entries may be unsorted within a row and may
 * repeat a column (they add up); rows may be empty.
 *
 *   rows, cols       >= 0 and < 2^31 - 1 (argument errors -1, -2)
 *   nnz              number of entries, 0 <= nnz < 2^31 (-3); must equal
 *                    row_offsets[rows]
 *   row_offsets      device, rows + 1 int32, row_offsets[0] = 0, nondecreasing (-4)
 *   column_indices   device, nnz int32 in [0, cols) (-5)
 *   values           device, nnz float (-6)
 *   alpha, beta      HOST pointers to float (-7, -9).  beta == 0: y is not
 *                    read.  alpha == 0 or nnz == 0: A and x are not read.
 *   x                device, cols float (-8)
 *   y                device, rows float, in/out (-10); must not overlap the
 *                    other arrays (DGA_ERR_OVERLAP)
 *   workspace        device scratch of dga_spmv_csr_workspace_size(rows, nnz)
 *                    bytes (-11 if NULL with workspace_bytes > 0,
 *                    DGA_ERR_WORKSPACE if smaller): one row index and one
 *                    partial sum per CTA, for rows that cross CTAs
 * Work is split evenly over rows + nnz whatever the row lengths.  Malformed
 * arrays never cause an access outside them: out-of-range column indices and
 * offsets are skipped or clamped and the next dga_sync_status() returns
 * DGA_ERR_BAD_INDEX.  Enqueued on `stream`; 2 kernel launches (1 when no
 * entry is read).
 */
int dga_spmv_csr(int64_t rows, int64_t cols, int64_t nnz, const int32_t* row_offsets,
                 const int32_t* column_indices, const float* values, const float* alpha,
                 const float* x, const float* beta, float* y, void* workspace,
                 size_t workspace_bytes, dga_stream_t stream);

/* Bytes of workspace dga_spmv_csr needs for rows and nnz on the current device
 * (152 SMs assumed when no device can be queried); 0 for rows <= 0. */
size_t dga_spmv_csr_workspace_size(int64_t rows, int64_t nnz);

/* Library version: major*10000 + minor*100 + patch. */
int dga_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DGA_H_ */
