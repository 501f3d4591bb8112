// FP32 FMA-rate probe: the denominator check for the SIMT GEMM's roofline
// (and, below it, the INT8 instruction-rate probe).
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

// INT8 instruction-rate probe: the legacy integer tensor instruction that
// an exact INT8 GEMM could be built on instead of the bf16 encoding, timed at
// its best (independent accumulator chains, operands already in registers).
// Every lane of warp w holds A bytes c = w % 5 + 1 and B bytes -2, so each
// m16n8k32 step adds 32 * c * (-2) to every accumulator element whatever the
// fragment layout, and a thread's sum over its 8 x 4 accumulators after
// `iters` steps of all 8 chains is -2048 * c * iters: the result shows the
// work was done.
constexpr int kMmaChains = 8;

__global__ void __launch_bounds__(kProbeThreads)
int8_mma_probe_kernel(int64_t iters, int32_t* out) {
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const uint32_t c = static_cast<uint32_t>(warp % 5) + 1;
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * c;
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = 0xFEFEFEFEu;  // bytes -2
    int32_t acc[kMmaChains][4];
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = 0;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kMmaChains; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    int32_t s = 0;
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) s += acc[j][i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

cudaError_t int8_mma_probe_launch(int64_t iters, int32_t* out, int sm_count, double* ops,
                                  cudaStream_t stream) {
    const int grid = sm_count * kProbeCtasPerSm;
    // per warp and iteration kMmaChains m16n8k32 steps of 2 * 16 * 8 * 32 ops
    *ops = static_cast<double>(grid) * (kProbeThreads / 32) * static_cast<double>(iters) *
           kMmaChains * (2.0 * 16 * 8 * 32);
    int8_mma_probe_kernel<<<grid, kProbeThreads, 0, stream>>>(iters, out);
    return cudaGetLastError();
}

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
