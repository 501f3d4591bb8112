// FP32 FMA-rate probe: the denominator check for the SIMT GEMM's roofline.
//
// The roofline of "Matrix multiplication: arithmetic intensity, tiling and
// Tensor Core" (section 5.1) bounds a compute-bound kernel by the chip's
// arithmetic peak.  For the FP32 SIMT path that peak is derived as
// SMs x 128 FP32 lanes x 2 FLOP x SM clock; this kernel measures the rate
// the FMA pipe actually sustains, once with scalar fmaf and once with the
// packed fma.rn.f32x2 the SIMT mainloop issues, so the derived figure can be
// checked against what the hardware does.
//
// Each thread runs kChains independent accumulator chains (enough to hide the
// FMA latency at 8 warps per scheduler), every step of every chain one fused
// multiply-add (or one packed pair).  The multiplier is just above 1 and the
// addend small, so the values stay normal and finite for any iteration count
// the entry point accepts.
#include <cstdint>

#include "dga_internal.h"

namespace dga {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 4;
constexpr int kChains = 8;
constexpr int kFmaPerIter = 64;  // per thread and loop iteration, both kernels

__global__ void __launch_bounds__(kProbeThreads)
fma_probe_kernel(int64_t iters, float* out) {
    float acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = fmaf(1e-3f, static_cast<float>(threadIdx.x + c), 1.0f);
    const float m = 1.0000001f, b = 1e-7f;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < kFmaPerIter / kChains; ++u)
#pragma unroll
            for (int c = 0; c < kChains; ++c) acc[c] = fmaf(acc[c], m, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kProbeThreads)
fma2_probe_kernel(int64_t iters, float* out) {
    uint64_t acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        const float lo = fmaf(1e-3f, static_cast<float>(threadIdx.x + c), 1.0f), hi = lo + 0.5f;
        asm("mov.b64 %0, {%1, %2};" : "=l"(acc[c]) : "f"(lo), "f"(hi));
    }
    uint64_t m, b;
    asm("mov.b64 %0, {%1, %1};" : "=l"(m) : "f"(1.0000001f));
    asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(1e-7f));
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < kFmaPerIter / (2 * kChains); ++u)
#pragma unroll
            for (int c = 0; c < kChains; ++c)
                asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[c]) : "l"(m), "l"(b));
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[c]));
        s += lo + hi;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

int64_t fma_probe_out_floats(int sm_count) {
    return static_cast<int64_t>(sm_count) * kProbeCtasPerSm * kProbeThreads;
}

cudaError_t fma_probe_launch(int packed, int64_t iters, float* out, int sm_count, double* flops,
                             cudaStream_t stream) {
    const int grid = sm_count * kProbeCtasPerSm;
    // both kernels do kFmaPerIter FMAs per thread and iteration (a packed
    // step counts as two), 2 FLOP each
    *flops = 2.0 * static_cast<double>(grid) * kProbeThreads * static_cast<double>(iters) * kFmaPerIter;
    if (packed)
        fma2_probe_kernel<<<grid, kProbeThreads, 0, stream>>>(iters, out);
    else
        fma_probe_kernel<<<grid, kProbeThreads, 0, stream>>>(iters, out);
    return cudaGetLastError();
}

}  // namespace dga
