// Counter-calibration probe: the naive GEMM of "GEMM optimisation, part 0",
// section 2 (one thread per output element, C(i, j) accumulated over k from
// A(i, k) * B(k, j), all three row-major and contiguous), launched in blocks
// of 16 x 16 threads with the block's x along the columns of C.  It belongs
// to no GEMM path of the library: it exists so that the hardware counters
// the profiles rest on can be checked against the figures that page prints
// for this very kernel at 2048^3 (section 2.3: one load request per warp per
// load instruction, 2 * 2048^3 / 32 = 536,870,912 requests; two 32-byte
// sectors per request).
#include <cstdint>

#include "dga_internal.h"

namespace dga {
namespace {

constexpr int kNaiveBlock = 16;

__global__ void naive_sgemm_kernel(int64_t M, int64_t N, int64_t K, const float* __restrict__ A,
                                   const float* __restrict__ B, float* __restrict__ C) {
    const int64_t col = static_cast<int64_t>(blockIdx.x) * kNaiveBlock + threadIdx.x;
    const int64_t row = static_cast<int64_t>(blockIdx.y) * kNaiveBlock + threadIdx.y;
    if (row >= M || col >= N) return;
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k) acc = fmaf(A[row * K + k], B[k * N + col], acc);
    C[row * N + col] = acc;
}

}  // namespace

cudaError_t naive_probe_launch(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                               float* C, cudaStream_t stream) {
    const dim3 block(kNaiveBlock, kNaiveBlock);
    const dim3 grid(static_cast<unsigned>((N + kNaiveBlock - 1) / kNaiveBlock),
                    static_cast<unsigned>((M + kNaiveBlock - 1) / kNaiveBlock));
    naive_sgemm_kernel<<<grid, block, 0, stream>>>(M, N, K, A, B, C);
    return cudaGetLastError();
}

}  // namespace dga
