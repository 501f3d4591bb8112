// gemm_generic.cu -- the kernel family that accepts every argument set the
// ABI allows: any supported dtype pair, either B layout, any leading
// dimension and any pointer alignment.  It keeps the API total for shapes the
// fast families reject (TMA needs 16-byte strides, the SIMT kernel float4
// loads); it is still GPU code, never a CPU fallback.
//
// Structure: the shared-memory tiled GEMM of "AI Programming: Matrix
// Product", section "Shared Memory Tiling" -- a T x T output tile per block,
// A and B staged through shared memory one K-slice at a time, out-of-range
// elements loaded as zero, stores masked -- widened here with a 2 x 2
// register tile per thread (32 x 32 outputs per 16 x 16 block), a
// layout-aware A and B loads, and the dtype-generic epilogue (with the
// optional bias row of the fully-connected layer, same page, section
// "Fully-connected layer").  K == 0 or alpha == 0 skips the loads entirely
// (C <- beta*C + bias; beta == 0 writes without reading C).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dga_internal.h"
#include "epilogue.cuh"

namespace dga {
namespace {

constexpr int kT = 32;       // output tile edge
constexpr int kTK = 16;      // K-slice per shared-memory stage
constexpr int kThreads = 16;  // block is kThreads x kThreads; 2 x 2 outputs each

template <typename T> struct InT;
template <> struct InT<float> {
    using Acc = float;
    __device__ __forceinline__ static float get(const float* p) { return *p; }
};
template <> struct InT<__nv_bfloat16> {
    using Acc = float;
    __device__ __forceinline__ static float get(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
};
template <> struct InT<__half> {
    using Acc = float;
    __device__ __forceinline__ static float get(const __half* p) { return __half2float(*p); }
};
template <> struct InT<int8_t> {
    using Acc = int32_t;
    __device__ __forceinline__ static int32_t get(const int8_t* p) { return *p; }
};

struct Params {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    void* C;
    int64_t ldc;
    const void* bias;  // N output-type elements added to every row, or null
    int layout_a, layout_b;
    float alpha_f, beta_f;
    int32_t alpha_i, beta_i;
    int skip_product;  // alpha == 0 or K == 0
};

template <typename TAcc, typename TOut>
__device__ __forceinline__ void finish(const Params& p, TAcc acc, int64_t r, int64_t c);

template <>
__device__ __forceinline__ void finish<int32_t, int32_t>(const Params& p, int32_t acc,
                                                         int64_t r, int64_t c) {
    int32_t* C = static_cast<int32_t*>(p.C) + r * p.ldc + c;
    int32_t old = p.beta_i != 0 ? *C : 0;
    int32_t v = axpby_i32(p.alpha_i, acc, p.beta_i, old);
    if (p.bias) v = static_cast<int32_t>(static_cast<uint32_t>(v) +
                                         static_cast<uint32_t>(static_cast<const int32_t*>(p.bias)[c]));
    *C = v;
}

template <typename TAcc, typename TOut>
__device__ __forceinline__ void finish(const Params& p, TAcc acc, int64_t r, int64_t c) {
    TOut* C = static_cast<TOut*>(p.C) + r * p.ldc + c;
    float old = p.beta_f != 0.0f ? OutT<TOut>::load(C) : 0.0f;
    float v = axpby(p.alpha_f, static_cast<float>(acc), p.beta_f, old);
    if (p.bias) v += OutT<TOut>::load(static_cast<const TOut*>(p.bias) + c);
    OutT<TOut>::store(C, v);
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads* kThreads) gemm_generic_kernel(Params p) {
    using Acc = typename InT<TIn>::Acc;
    __shared__ Acc As[kTK][kT + 1];  // As[k][m]
    __shared__ Acc Bs[kTK][kT + 1];  // Bs[k][n]
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int tid = ty * kThreads + tx;
    const int64_t row0 = static_cast<int64_t>(blockIdx.y) * kT;
    const int64_t col0 = static_cast<int64_t>(blockIdx.x) * kT;
    const TIn* A = static_cast<const TIn*>(p.A);
    const TIn* B = static_cast<const TIn*>(p.B);

    Acc acc[2][2] = {};
    if (!p.skip_product) {
        for (int64_t k0 = 0; k0 < p.K; k0 += kTK) {
            // 32 x 16 elements of A and 16 x 32 of B; 256 threads, 2 each.
            for (int e = tid; e < kT * kTK; e += kThreads * kThreads) {
                int m, k;  // consecutive threads walk the contiguous direction of A
                if (p.layout_a == DGA_ROW_MAJOR) { m = e / kTK; k = e % kTK; }
                else { k = e / kT; m = e % kT; }
                int64_t gr = row0 + m, gk = k0 + k;
                const TIn* src = p.layout_a == DGA_ROW_MAJOR ? A + gr * p.lda + gk : A + gk * p.lda + gr;
                As[k][m] = (gr < p.M && gk < p.K) ? InT<TIn>::get(src) : Acc(0);
            }
            for (int e = tid; e < kT * kTK; e += kThreads * kThreads) {
                int k, n;
                if (p.layout_b == DGA_ROW_MAJOR) { k = e / kT; n = e % kT; }
                else { n = e / kTK; k = e % kTK; }
                int64_t gk = k0 + k, gc = col0 + n;
                const TIn* src = p.layout_b == DGA_ROW_MAJOR ? B + gk * p.ldb + gc
                                                             : B + gc * p.ldb + gk;
                Bs[k][n] = (gk < p.K && gc < p.N) ? InT<TIn>::get(src) : Acc(0);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kTK; ++k) {
                Acc a0 = As[k][ty], a1 = As[k][ty + kThreads];
                Acc b0 = Bs[k][tx], b1 = Bs[k][tx + kThreads];
                acc[0][0] += a0 * b0;
                acc[0][1] += a0 * b1;
                acc[1][0] += a1 * b0;
                acc[1][1] += a1 * b1;
            }
            __syncthreads();  // the next slice overwrites As/Bs
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            int64_t r = row0 + ty + i * kThreads, c = col0 + tx + j * kThreads;
            if (r < p.M && c < p.N) finish<Acc, TOut>(p, acc[i][j], r, c);
        }
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const Params& p, cudaStream_t s) {
    dim3 block(kThreads, kThreads);
    dim3 grid(static_cast<unsigned>((p.N + kT - 1) / kT), static_cast<unsigned>((p.M + kT - 1) / kT));
    gemm_generic_kernel<TIn, TOut><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool generic_supports(const GemmArgs& a) {
    // grid.y limit: 65535 tiles of 32 rows
    return (a.M + kT - 1) / kT <= 65535 && (a.N + kT - 1) / kT <= 0x7fffffff;
}

cudaError_t generic_launch(const GemmArgs& a, int* launches) {
    Params p{a.M, a.N, a.K, a.A, a.lda, a.B, a.ldb, a.C, a.ldc, a.bias, a.layout_a, a.layout_b,
             a.alpha_f, a.beta_f, a.alpha_i, a.beta_i, (a.K == 0 || alpha_is_zero(a)) ? 1 : 0};
    cudaError_t e = cudaErrorInvalidValue;
    // TF32 inputs are fp32 in memory; this family multiplies them exactly in
    // fp32, which is within the TF32 error bound
    if ((a.in_dtype == DGA_F32 || a.in_dtype == DGA_TF32) && a.out_dtype == DGA_F32)
        e = launch_typed<float, float>(p, a.stream);
    else if (a.in_dtype == DGA_BF16 && a.out_dtype == DGA_F32) e = launch_typed<__nv_bfloat16, float>(p, a.stream);
    else if (a.in_dtype == DGA_BF16 && a.out_dtype == DGA_BF16) e = launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a.stream);
    else if (a.in_dtype == DGA_F16 && a.out_dtype == DGA_F32) e = launch_typed<__half, float>(p, a.stream);
    else if (a.in_dtype == DGA_F16 && a.out_dtype == DGA_F16) e = launch_typed<__half, __half>(p, a.stream);
    else if (a.in_dtype == DGA_I8 && a.out_dtype == DGA_I32) e = launch_typed<int8_t, int32_t>(p, a.stream);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace dga
