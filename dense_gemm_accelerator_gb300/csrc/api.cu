// api.cu -- the C ABI of include/dga.h: argument checks, path selection, and
// the launch of the chosen kernel family on the caller's stream.
//
// The operation is BLAS GEMM, C <- alpha*A*B + beta*C ("AI Programming:
// Matrix Product", section "Dense matrix multiplication"), with row-major
// offsets row*ld + col (section "Row-major order").  BLAS conventions decide
// what the pages leave open: M == 0 or N == 0 is a no-op, K == 0 or
// alpha == 0 reads neither A nor B, beta == 0 never reads C, and invalid
// arguments are reported as -(their 1-based position).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "dga_internal.h"

namespace dga {
namespace {

thread_local int t_last_path = DGA_PATH_AUTO;
thread_local int t_last_launches = 0;
thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
cudaError_t g_dev_err[kMaxDevices];

bool pair_supported(int in, int out) {
    return (in == DGA_F32 && out == DGA_F32) || (in == DGA_BF16 && (out == DGA_F32 || out == DGA_BF16)) ||
           (in == DGA_F16 && (out == DGA_F32 || out == DGA_F16)) || (in == DGA_I8 && out == DGA_I32) ||
           (in == DGA_TF32 && out == DGA_F32);
}

size_t elem_size(int dt) {
    switch (dt) {
    case DGA_F32: case DGA_I32: case DGA_TF32: return 4;
    case DGA_BF16: case DGA_F16: return 2;
    case DGA_I8: return 1;
    default: return 0;
    }
}

// Byte range [lo, hi) that a rows x cols matrix with row stride ld occupies.
void span(const void* p, int64_t rows, int64_t cols, int64_t ld, size_t es, uintptr_t* lo,
          uintptr_t* hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * static_cast<int64_t>(es));
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// 1-based positions of the checked arguments in one entry point's list, so
// that argument errors come back as -(position) in that entry point's terms.
struct ArgPos {
    int M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ws;
};
constexpr ArgPos kPosEx{4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15};
constexpr ArgPos kPosGeneral{5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 17};

// Validates everything but the pointers' alignment; fills *g.  Without
// `with_pointers` (size queries), matrix pointers are neither required nor
// checked for overlap.
int check_args(const ArgPos& pos, dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
               dga_layout layout_b, int64_t M, int64_t N, int64_t K, const void* alpha,
               const void* A, int64_t lda, const void* B, int64_t ldb, const void* beta, void* C,
               int64_t ldc, const void* bias, void* ws, size_t ws_bytes, GemmArgs* g,
               bool with_pointers = true) {
    if (in_dtype < DGA_F32 || in_dtype > DGA_TF32 || out_dtype < DGA_F32 || out_dtype > DGA_TF32)
        return DGA_ERR_UNSUPPORTED;
    if (layout_a != DGA_ROW_MAJOR && layout_a != DGA_COL_MAJOR) return DGA_ERR_UNSUPPORTED;
    if (layout_b != DGA_ROW_MAJOR && layout_b != DGA_COL_MAJOR) return DGA_ERR_UNSUPPORTED;
    if (!pair_supported(in_dtype, out_dtype)) return DGA_ERR_UNSUPPORTED;
    if (M < 0) return -pos.M;
    if (N < 0) return -pos.N;
    if (K < 0) return -pos.K;
    if (!alpha) return -pos.alpha;
    if (!beta) return -pos.beta;
    g->in_dtype = in_dtype;
    g->out_dtype = out_dtype;
    g->layout_a = layout_a;
    g->layout_b = layout_b;
    g->M = M;
    g->N = N;
    g->K = K;
    if (in_dtype == DGA_I8) {
        std::memcpy(&g->alpha_i, alpha, sizeof(int32_t));
        std::memcpy(&g->beta_i, beta, sizeof(int32_t));
        g->alpha_f = static_cast<float>(g->alpha_i);
        g->beta_f = static_cast<float>(g->beta_i);
    } else {
        std::memcpy(&g->alpha_f, alpha, sizeof(float));
        std::memcpy(&g->beta_f, beta, sizeof(float));
        g->alpha_i = 0;
        g->beta_i = 0;
    }
    const bool reads_ab = with_pointers && M > 0 && N > 0 && K > 0 && !alpha_is_zero(*g);
    if (reads_ab && !A) return -pos.A;
    const int64_t min_lda = layout_a == DGA_ROW_MAJOR ? (K > 1 ? K : 1) : (M > 1 ? M : 1);
    if (lda < min_lda) return -pos.lda;
    if (reads_ab && !B) return -pos.B;
    const int64_t min_ldb = layout_b == DGA_ROW_MAJOR ? (N > 1 ? N : 1) : (K > 1 ? K : 1);
    if (ldb < min_ldb) return -pos.ldb;
    if (with_pointers && M > 0 && N > 0 && !C) return -pos.C;
    if (ldc < (N > 1 ? N : 1)) return -pos.ldc;
    if (ws_bytes > 0 && !ws) return -pos.ws;
    g->A = A;
    g->lda = lda;
    g->B = B;
    g->ldb = ldb;
    g->C = C;
    g->ldc = ldc;
    g->bias = bias;
    g->ws = ws;
    g->ws_bytes = ws_bytes;
    if (with_pointers && M > 0 && N > 0) {
        uintptr_t c0, c1;
        span(C, M, N, ldc, elem_size(out_dtype), &c0, &c1);
        if (bias) {
            uintptr_t v0, v1;
            span(bias, 1, N, N, elem_size(out_dtype), &v0, &v1);
            if (overlaps(c0, c1, v0, v1)) return DGA_ERR_OVERLAP;
        }
        if (reads_ab) {
            uintptr_t a0, a1, b0, b1;
            if (layout_a == DGA_ROW_MAJOR) span(A, M, K, lda, elem_size(in_dtype), &a0, &a1);
            else span(A, K, M, lda, elem_size(in_dtype), &a0, &a1);
            if (layout_b == DGA_ROW_MAJOR) span(B, K, N, ldb, elem_size(in_dtype), &b0, &b1);
            else span(B, N, K, ldb, elem_size(in_dtype), &b0, &b1);
            if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return DGA_ERR_OVERLAP;
        }
    }
    return DGA_OK;
}

// AUTO: the fastest family that accepts the arguments.
int choose_path(const GemmArgs& g) {
    if (g.K == 0 || alpha_is_zero(g)) return DGA_PATH_GENERIC;  // C <- beta*C only
    if (g.in_dtype == DGA_F32) return simt_supports(g) ? DGA_PATH_SIMT : DGA_PATH_GENERIC;
    if (g.in_dtype == DGA_BF16 || g.in_dtype == DGA_F16) {
        if (skinny_supports(g)) return DGA_PATH_SKINNY;
        if (tc_supports(g)) return DGA_PATH_TCGEN05;
        return DGA_PATH_GENERIC;
    }
    if (g.in_dtype == DGA_I8 || g.in_dtype == DGA_TF32)
        return tc_supports(g) ? DGA_PATH_TCGEN05 : DGA_PATH_GENERIC;
    return DGA_PATH_GENERIC;
}

bool path_accepts(int path, const GemmArgs& g) {
    const bool no_product = g.K == 0 || alpha_is_zero(g);
    switch (path) {
    case DGA_PATH_GENERIC: return generic_supports(g);
    case DGA_PATH_SIMT: return !no_product && simt_supports(g);
    case DGA_PATH_TCGEN05: return !no_product && tc_supports(g);
    case DGA_PATH_SKINNY: return !no_product && skinny_supports(g);
    default: return false;
    }
}

// Workspace the call cannot run without.
size_t workspace_required(int path, const GemmArgs& g) {
    return path == DGA_PATH_TCGEN05 ? tc_workspace_size(g) : 0;
}

// SM count of the current device for size queries made without a GPU: the
// real count when the device can be queried, else 152 (GB300).
int sm_count_or_default() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();  // clear the failed query
    return 152;
}

// Workspace the call would use if given: required bytes, plus for the SIMT
// and tensor-core paths the optional bytes of their split last waves.
size_t workspace_wanted(int path, const GemmArgs& g) {
    if (path == DGA_PATH_SIMT) return simt_workspace_size(g, sm_count_or_default());
    if (path == DGA_PATH_TCGEN05) return tc_workspace_wanted(g, sm_count_or_default());
    return workspace_required(path, g);
}

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return DGA_ERR_CUDA;
}

}  // namespace

int note_cuda_error(cudaError_t e) { return fail_cuda(e); }

cudaError_t current_device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_dev_once[dev], [dev] {
        DeviceInfo d{};
        d.ordinal = dev;
        cudaError_t err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        g_dev[dev] = d;
        g_dev_err[dev] = err;
    });
    *out = g_dev[dev];
    return g_dev_err[dev];
}

}  // namespace dga

using namespace dga;

namespace {

int gemm_impl(const ArgPos& pos, dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
              dga_layout layout_b, int64_t M, int64_t N, int64_t K, const void* alpha,
              const void* A, int64_t lda, const void* B, int64_t ldb, const void* beta, void* C,
              int64_t ldc, const void* bias, void* workspace, size_t workspace_bytes,
              dga_path path, dga_stream_t stream) {
    GemmArgs g{};
    int st = check_args(pos, in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B,
                        ldb, beta, C, ldc, bias, workspace, workspace_bytes, &g);
    if (st != DGA_OK) return st;
    g.stream = reinterpret_cast<cudaStream_t>(stream);
    t_last_path = DGA_PATH_AUTO;
    t_last_launches = 0;
    if (M == 0 || N == 0) return DGA_OK;

    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev.major != 10 || dev.minor != 3) return DGA_ERR_DEVICE;

    const int chosen = path == DGA_PATH_AUTO ? choose_path(g) : static_cast<int>(path);
    if (!path_accepts(chosen, g)) return DGA_ERR_PATH;
    if (workspace_bytes < workspace_required(chosen, g)) return DGA_ERR_WORKSPACE;

    int launches = 0;
    switch (chosen) {
    case DGA_PATH_GENERIC: e = generic_launch(g, &launches); break;
    case DGA_PATH_SIMT: e = simt_launch(g, dev, &launches); break;
    case DGA_PATH_SKINNY: e = skinny_launch(g, dev, &launches); break;
    case DGA_PATH_TCGEN05: e = tc_launch(g, dev, &launches); break;
    default: return DGA_ERR_PATH;
    }
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_path = chosen;
    t_last_launches = launches;
    return DGA_OK;
}

}  // namespace

extern "C" {

int dga_gemm_general(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
                     dga_layout layout_b, int64_t M, int64_t N, int64_t K, const void* alpha,
                     const void* A, int64_t lda, const void* B, int64_t ldb, const void* beta,
                     void* C, int64_t ldc, const void* bias, void* workspace,
                     size_t workspace_bytes, dga_path path, dga_stream_t stream) {
    if (path < DGA_PATH_AUTO || path > DGA_PATH_SKINNY) return -19;
    return gemm_impl(kPosGeneral, in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, A, lda,
                     B, ldb, beta, C, ldc, bias, workspace, workspace_bytes, path, stream);
}

int dga_gemm_ex(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b, int64_t M, int64_t N,
                int64_t K, const void* alpha, const void* A, int64_t lda, const void* B,
                int64_t ldb, const void* beta, void* C, int64_t ldc, void* workspace,
                size_t workspace_bytes, dga_path path, dga_stream_t stream) {
    if (path < DGA_PATH_AUTO || path > DGA_PATH_SKINNY) return -17;
    return gemm_impl(kPosEx, in_dtype, out_dtype, DGA_ROW_MAJOR, layout_b, M, N, K, alpha, A, lda,
                     B, ldb, beta, C, ldc, nullptr, workspace, workspace_bytes, path, stream);
}

int dga_gemm(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b, int64_t M, int64_t N,
             int64_t K, const void* alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
             const void* beta, void* C, int64_t ldc, void* workspace, size_t workspace_bytes,
             dga_stream_t stream) {
    return dga_gemm_ex(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                       workspace, workspace_bytes, DGA_PATH_AUTO, stream);
}

int dga_sum_rows(dga_dtype dtype, int64_t rows, int64_t cols, const void* G, int64_t ldg,
                 float* out, dga_stream_t stream) {
    if (dtype != DGA_F32 && dtype != DGA_BF16 && dtype != DGA_F16) return DGA_ERR_UNSUPPORTED;
    if (rows < 0) return -2;
    if (cols < 0) return -3;
    if (cols == 0) return DGA_OK;
    if (rows > 0 && !G) return -4;
    if (ldg < (cols > 1 ? cols : 1)) return -5;
    if (!out) return -6;
    cudaError_t e = sum_rows_launch(dtype, rows, cols, G, ldg, out,
                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DGA_OK : fail_cuda(e);
}

namespace {

// The workspace query, for the bytes a call would use (wanted) or only those
// it cannot run without (required).
size_t workspace_query(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
                       dga_layout layout_b, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, dga_path path, bool required_only) {
    GemmArgs g{};
    const float one = 1.0f;
    const int32_t one_i = 1;
    const void* alpha = in_dtype == DGA_I8 ? static_cast<const void*>(&one_i) : &one;
    if (check_args(kPosGeneral, in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, nullptr,
                   lda, nullptr, ldb, alpha, nullptr, ldc, nullptr, nullptr, 0, &g,
                   /*with_pointers=*/false) != DGA_OK)
        return 0;
    if (M == 0 || N == 0 || K == 0) return 0;
    // Pointer-free query: operands are assumed 16-byte aligned.
    static const char aligned16[16] __attribute__((aligned(16))) = {};
    int chosen = static_cast<int>(path);
    if (path == DGA_PATH_AUTO) {
        GemmArgs probe = g;
        probe.A = aligned16;
        probe.B = aligned16;
        chosen = choose_path(probe);
    }
    return required_only ? workspace_required(chosen, g) : workspace_wanted(chosen, g);
}

}  // namespace

size_t dga_gemm_general_workspace_size(dga_dtype in_dtype, dga_dtype out_dtype,
                                       dga_layout layout_a, dga_layout layout_b, int64_t M,
                                       int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                       int64_t ldc, dga_path path) {
    return workspace_query(in_dtype, out_dtype, layout_a, layout_b, M, N, K, lda, ldb, ldc, path,
                           false);
}

size_t dga_gemm_workspace_size(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b,
                               int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldc, dga_path path) {
    return dga_gemm_general_workspace_size(in_dtype, out_dtype, DGA_ROW_MAJOR, layout_b, M, N, K,
                                           lda, ldb, ldc, path);
}

int dga_select_path(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_b, int64_t M,
                    int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                    const void* C, int64_t ldc) {
    GemmArgs g{};
    const float one = 1.0f;
    const int32_t one_i = 1;
    const void* alpha = in_dtype == DGA_I8 ? static_cast<const void*>(&one_i) : &one;
    int st = check_args(kPosEx, in_dtype, out_dtype, DGA_ROW_MAJOR, layout_b, M, N, K, alpha, A,
                        lda, B, ldb, alpha, const_cast<void*>(C), ldc, nullptr, nullptr, 0, &g);
    if (st != DGA_OK) return st < 0 ? st : -st;
    return choose_path(g);
}

size_t dga_spmv_csr_workspace_size(int64_t rows, int64_t nnz) {
    if (rows <= 0 || nnz < 0) return 0;
    return spmv_workspace_size(rows, nnz, sm_count_or_default());
}

int dga_spmv_csr(int64_t rows, int64_t cols, int64_t nnz, const int32_t* row_offsets,
                 const int32_t* column_indices, const float* values, const float* alpha,
                 const float* x, const float* beta, float* y, void* workspace,
                 size_t workspace_bytes, dga_stream_t stream) {
    if (rows < 0 || rows >= (int64_t(1) << 31) - 1) return -1;
    if (cols < 0 || cols >= (int64_t(1) << 31)) return -2;
    if (nnz < 0 || nnz >= (int64_t(1) << 31)) return -3;
    if (!alpha) return -7;
    if (!beta) return -9;
    t_last_path = DGA_PATH_AUTO;
    t_last_launches = 0;
    if (rows == 0) return DGA_OK;
    if (!row_offsets) return -4;
    const float a = *alpha, b = *beta;
    const bool reads_a = a != 0.0f && nnz > 0;
    if (reads_a && !column_indices) return -5;
    if (reads_a && !values) return -6;
    if (reads_a && !x) return -8;
    if (!y) return -10;
    if (workspace_bytes > 0 && !workspace) return -11;
    // y must not overlap the arrays it is computed from
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(y), y1 = y0 + static_cast<uintptr_t>(rows) * 4;
    auto hits = [&](const void* q, int64_t bytes) {
        const uintptr_t q0 = reinterpret_cast<uintptr_t>(q);
        return q && bytes > 0 && overlaps(y0, y1, q0, q0 + static_cast<uintptr_t>(bytes));
    };
    if (hits(row_offsets, (rows + 1) * 4) || (reads_a && (hits(column_indices, nnz * 4) ||
                                                          hits(values, nnz * 4) || hits(x, cols * 4))))
        return DGA_ERR_OVERLAP;
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev.major != 10 || dev.minor != 3) return DGA_ERR_DEVICE;
    if (reads_a && workspace_bytes < spmv_workspace_size(rows, nnz, dev.sm_count))
        return DGA_ERR_WORKSPACE;
    int launches = 0;
    e = spmv_launch(rows, cols, nnz, row_offsets, column_indices, values, a, x, b, y, workspace,
                    workspace_bytes, dev, reinterpret_cast<cudaStream_t>(stream), &launches);
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_launches = launches;
    return DGA_OK;
}

int dga_last_path(void) { return t_last_path; }

int dga_last_launch_count(void) { return t_last_launches; }

int dga_sync_status(dga_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    int st = 0, st_skinny = 0, st_spmv = 0;
    e = tc_status_take(&st);
    if (e == cudaSuccess) e = skinny_status_take(&st_skinny);
    if (e == cudaSuccess) e = spmv_status_take(&st_spmv);
    if (e != cudaSuccess) return fail_cuda(e);
    if (st != 0 || st_skinny != 0) return DGA_ERR_DEVICE_TIMEOUT;
    return st_spmv != 0 ? DGA_ERR_BAD_INDEX : DGA_OK;
}

int dga_last_cuda_error(void) { return t_last_cuda_error; }

int dga_selftest_bounded_wait(int64_t limit_ns, dga_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > 2000000000) return -1;
    cudaError_t e = tc_selftest_wait(static_cast<uint64_t>(limit_ns),
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DGA_OK : fail_cuda(e);
}

int64_t dga_probe_fp32_fma_out_floats(void) { return fma_probe_out_floats(sm_count_or_default()); }

int dga_probe_fp32_fma(int packed, int64_t iters, float* out, int64_t out_floats, double* flops,
                       dga_stream_t stream) {
    if (packed != 0 && packed != 1) return -1;
    if (iters < 1 || iters > (int64_t{1} << 20)) return -2;
    if (out == nullptr) return -3;
    if (flops == nullptr) return -5;
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev.major != 10 || dev.minor != 3) return DGA_ERR_DEVICE;
    if (out_floats < fma_probe_out_floats(dev.sm_count)) return -4;
    e = fma_probe_launch(packed, iters, out, dev.sm_count, flops,
                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_launches = 1;
    return DGA_OK;
}

int dga_probe_int8_mma(int64_t iters, int32_t* out, int64_t out_ints, double* ops,
                       dga_stream_t stream) {
    if (iters < 1 || iters > (int64_t{1} << 17)) return -1;
    if (out == nullptr) return -2;
    if (ops == nullptr) return -4;
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev.major != 10 || dev.minor != 3) return DGA_ERR_DEVICE;
    if (out_ints < fma_probe_out_floats(dev.sm_count)) return -3;
    e = int8_mma_probe_launch(iters, out, dev.sm_count, ops, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_launches = 1;
    return DGA_OK;
}

int dga_probe_naive_sgemm(int64_t M, int64_t N, int64_t K, const float* A, const float* B, float* C,
                          dga_stream_t stream) {
    constexpr int64_t kMaxElems = int64_t{1} << 31;  // every index stays below 2^31
    if (M < 1 || M > 65536) return -1;
    if (N < 1 || N > 65536) return -2;
    if (K < 1 || K > 65536 || M * K >= kMaxElems || K * N >= kMaxElems || M * N >= kMaxElems)
        return -3;
    if (A == nullptr) return -4;
    if (B == nullptr) return -5;
    if (C == nullptr) return -6;
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev.major != 10 || dev.minor != 3) return DGA_ERR_DEVICE;
    e = naive_probe_launch(M, N, K, A, B, C, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_launches = 1;
    return DGA_OK;
}

const char* dga_status_string(int status) {
    if (status < 0) return "invalid argument (the negated value is its 1-based position)";
    switch (status) {
    case DGA_OK: return "ok";
    case DGA_ERR_UNSUPPORTED: return "unsupported dtype pair or layout";
    case DGA_ERR_CUDA: return "a CUDA call failed";
    case DGA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
    case DGA_ERR_PATH: return "the forced kernel family cannot run these arguments";
    case DGA_ERR_WORKSPACE: return "workspace smaller than dga_gemm_workspace_size()";
    case DGA_ERR_OVERLAP: return "C overlaps A or B";
    case DGA_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case DGA_ERR_BAD_INDEX: return "a CSR index or row offset was out of range (reported by dga_sync_status)";
    default: return "unknown status";
    }
}

int dga_version(void) { return 310; }  // 0.3.1: split last waves on the tensor cores (INT8 included)

}  // extern "C"

size_t dga::workspace_required_bytes(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
                                     dga_layout layout_b, int64_t M, int64_t N, int64_t K,
                                     int64_t lda, int64_t ldb, int64_t ldc, dga_path path) {
    return workspace_query(in_dtype, out_dtype, layout_a, layout_b, M, N, K, lda, ldb, ldc, path,
                           true);
}
