// dga_internal.h -- host-side declarations shared by the library's
// translation units (one per kernel family) and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "dga.h"

namespace dga {

// One validated GEMM call.  alpha/beta are kept both as float (floating-point
// inputs) and as int32 (INT8 inputs); only the one matching in_dtype is used.
struct GemmArgs {
    int in_dtype, out_dtype, layout_a, layout_b;
    int64_t M, N, K;
    float alpha_f, beta_f;
    int32_t alpha_i, beta_i;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    void* C;
    int64_t ldc;
    const void* bias;  // N elements of the output type (int32 for INT8), or null
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

struct DeviceInfo {
    int ordinal;
    int sm_count;
    int major, minor;
    int max_smem_optin;  // bytes of dynamic shared memory one block may opt into
};

// Records `e` as this host thread's last CUDA error; returns DGA_ERR_CUDA.
int note_cuda_error(cudaError_t e);

// Properties of the current device (queried once per device).
cudaError_t current_device_info(DeviceInfo* out);

inline bool aligned(const void* p, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(p) % bytes) == 0;
}

inline bool alpha_is_zero(const GemmArgs& a) {
    return a.in_dtype == DGA_I8 ? a.alpha_i == 0 : a.alpha_f == 0.0f;
}

// ---- kernel families: supports() says whether the family can run the
// arguments; launch() enqueues its kernels and adds their count to *launches.

// Column sums of a rows x cols matrix into fp32 (the bias gradient).
cudaError_t sum_rows_launch(int dtype, int64_t rows, int64_t cols, const void* G, int64_t ldg,
                            float* out, cudaStream_t stream);

bool generic_supports(const GemmArgs& a);
cudaError_t generic_launch(const GemmArgs& a, int* launches);

bool simt_supports(const GemmArgs& a);
// Optional workspace: with this many bytes the last wave is split along K.
size_t simt_workspace_size(const GemmArgs& a, int sm_count);
cudaError_t simt_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches);

bool skinny_supports(const GemmArgs& a);
cudaError_t skinny_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches);
// Reads and clears this device's skinny-path status word.
cudaError_t skinny_status_take(int* status);

// CSR sparse matrix-vector product (validated arguments; alpha, beta by value).
size_t spmv_workspace_size(int64_t rows, int64_t nnz, int sm_count);
cudaError_t spmv_launch(int64_t rows, int64_t cols, int64_t nnz, const int32_t* row_offsets,
                        const int32_t* column_indices, const float* values, float alpha,
                        const float* x, float beta, float* y, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t stream, int* launches);
// Reads and clears this device's SpMV status word (non-zero: malformed CSR arrays).
cudaError_t spmv_status_take(int* status);

// FP32 FMA-rate probe (measurement only): floats of `out` one launch writes,
// and the launch itself (*flops receives the FLOPs it performs).
int64_t fma_probe_out_floats(int sm_count);  // also the int32s of the INT8 probe
cudaError_t int8_mma_probe_launch(int64_t iters, int32_t* out, int sm_count, double* ops,
                                  cudaStream_t stream);
cudaError_t fma_probe_launch(int packed, int64_t iters, float* out, int sm_count, double* flops,
                             cudaStream_t stream);

// Naive GEMM for counter calibration (measurement only): C = A * B, all
// row-major and contiguous, one thread per output in 16 x 16 blocks.
cudaError_t naive_probe_launch(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                               float* C, cudaStream_t stream);

bool tc_supports(const GemmArgs& a);
size_t tc_workspace_size(const GemmArgs& a);
// tc_workspace_size plus what the split last wave can use (optional)
size_t tc_workspace_wanted(const GemmArgs& a, int sm_count);
// The workspace a call cannot run without (dga_gemm_general_workspace_size
// reports this plus the optional bytes); 0 for invalid arguments.
size_t workspace_required_bytes(dga_dtype in_dtype, dga_dtype out_dtype, dga_layout layout_a,
                                dga_layout layout_b, int64_t M, int64_t N, int64_t K, int64_t lda,
                                int64_t ldb, int64_t ldc, dga_path path);
cudaError_t tc_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches);
// Launches a kernel whose bounded wait runs out after limit_ns (self-test).
cudaError_t tc_selftest_wait(uint64_t limit_ns, cudaStream_t stream);
// Reads and clears this device's tcgen05 status word (non-zero: a wait expired).
cudaError_t tc_status_take(int* status);

}  // namespace dga
