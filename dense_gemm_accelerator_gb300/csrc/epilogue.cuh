// epilogue.cuh -- the fused output step shared by every kernel family:
//     out = alpha * acc + beta * c_old      (c_old is read only when beta != 0)
// computed in fp32 (int32 with wrap-around for INT8), then converted to the
// output type with round-to-nearest-even, and stored only where the element
// exists (row < M, col < N), so edge tiles never touch memory outside C.
// The BLAS update C <- alpha*A*B + beta*C is the one of "AI Programming:
// Matrix Product", section "Dense matrix multiplication"; the masked store
// follows its "Shared Memory Tiling" kernel, which guards the final write
// with row < m && col < n.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace dga {

template <typename T> struct OutT;

template <> struct OutT<float> {
    __device__ __forceinline__ static float load(const float* p) { return *p; }
    __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
};
template <> struct OutT<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};
template <> struct OutT<__half> {
    __device__ __forceinline__ static float load(const __half* p) { return __half2float(*p); }
    __device__ __forceinline__ static void store(__half* p, float v) { *p = __float2half_rn(v); }
};

// alpha*acc + beta*c in fp32: one rounding for alpha*acc, one fused for beta*c.
__device__ __forceinline__ float axpby(float alpha, float acc, float beta, float c) {
    return fmaf(beta, c, alpha * acc);
}

// The same in int32 two's complement, wrapping mod 2^32.
__device__ __forceinline__ int32_t axpby_i32(int32_t alpha, int32_t acc, int32_t beta,
                                             int32_t c) {
    uint32_t r = static_cast<uint32_t>(alpha) * static_cast<uint32_t>(acc) +
                 static_cast<uint32_t>(beta) * static_cast<uint32_t>(c);
    return static_cast<int32_t>(r);
}

}  // namespace dga
