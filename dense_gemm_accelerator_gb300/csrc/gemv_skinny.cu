// gemv_skinny.cu -- the bandwidth-bound path for skinny products
//     Y[M, N] = alpha * X[M, K] * W[N, K]^T + beta * Y,   M <= 16,
// i.e. dga_gemm with A = X (row-major), B column-major (W stored N x K, the
// Linear-layer weight layout of "AI Programming: Matrix Product", section
// "Fully-connected layer") and C = Y.
//
// Why a separate path: a GEMV moves 2 bytes of weight per multiply-add, so no
// amount of arithmetic speed helps; the time is the weight's bytes divided
// by HBM bandwidth ("Matrix multiplication: arithmetic intensity, tiling and
// Tensor Core", section 5.1, the matrix-vector row of its table, and section
// 5.6).  The design therefore only has to (1) read every weight byte exactly
// once, with enough loads in flight to saturate HBM, and (2) keep the
// arithmetic off the critical path.
//
//  * Each weight element is loaded once, 16 bytes per lane, with
//    ld.global.nc.L1::no_allocate (streamed, never re-read) and an L2
//    prefetch size of 256 bytes, so DRAM sees whole 256-byte requests for
//    rows that a warp walks 64 bytes at a time.
//  * The loads of several K steps are kept in flight per warp (a software
//    pipeline over a register ring), since the whole kernel is a single
//    pass over the weight.
//  * The M <= 16 activation rows are the "B" operand of an mma.sync
//    m16n8k16 (fp32 accumulate) and the weight rows its "A" operand, so a
//    warp computes 16 weight rows x 8 activation rows per instruction; the
//    FP32 FMA pipe alone could not keep up at M = 16 (2 M FLOP per weight
//    element at ~7 TB/s is ~110 TFLOP/s).
//  * No shuffles: a lane loads 8 consecutive k of one weight row and the same
//    8 k of one activation row.  The dot product over k does not depend on
//    the order of k, so these 8 values are fed to two MMAs as k-slots
//    {2t, 2t+1, 2t+8, 2t+9} (t = lane % 4) -- the same permutation on both
//    operands, hence the same sum.
//  * A CTA owns RT*16 weight rows; its warps split K, and the partial tiles
//    are summed in shared memory before the fused alpha/beta epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dga_internal.h"
#include "epilogue.cuh"

namespace dga {
namespace {

struct Params {
    int64_t M, N, K;
    const void* X;
    int64_t ldx;
    const void* W;
    int64_t ldw;
    void* Y;
    int64_t ldy;
    float alpha, beta;
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_cached(const void* p) {
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (kBf16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// One 32-element K step of a warp: RT weight tiles (two 16-byte loads per
// lane each: rows g and g+8) and MT activation tiles (one load per lane).
template <int RT, int MT>
struct Step {
    uint4 w[RT][2];
    uint4 x[MT];
};

// MT = number of 8-row activation tiles (1 for M <= 8, 2 for M <= 16);
// RT = 16-row weight tiles per CTA; WARPS split K; PF = K steps of loads
// kept in flight per warp (software pipeline depth).
template <bool kBf16, int MT, typename TOut, int RT, int WARPS, int PF>
__global__ void __launch_bounds__(WARPS * 32) skinny_kernel(Params p) {
    __shared__ float red[WARPS][RT * 16][MT * 8 + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * (RT * 16);

    // This warp's K range, in whole 32-element steps.
    const int64_t steps = (p.K + 31) / 32;
    const int64_t per_warp = (steps + WARPS - 1) / WARPS;
    const int64_t s_begin = warp * per_warp;
    const int64_t s_end = min(steps, s_begin + per_warp);

    const char* W = static_cast<const char*>(p.W);
    const char* X = static_cast<const char*>(p.X);
    // Row pointers (clamped when the row does not exist; such loads are skipped).
    const char* wrow[RT][2];
    bool wok[RT][2];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + r * 16 + g + h * 8;
            wok[r][h] = n < p.N;
            wrow[r][h] = W + (wok[r][h] ? n : 0) * p.ldw * 2;
        }
    const char* xrow[MT];
    bool xok[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int64_t row = m * 8 + g;
        xok[m] = row < p.M;
        xrow[m] = X + (xok[m] ? row : 0) * p.ldx * 2;
    }

    float acc[RT][MT][4];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][m][i] = 0.0f;

    const uint4 zero = make_uint4(0, 0, 0, 0);
    auto load = [&](Step<RT, MT>& st, int64_t s) {
        const int64_t k = s * 32 + t * 8;  // this lane's 8 consecutive k (K % 8 == 0)
        const bool kok = s < s_end && k < p.K;
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                st.w[r][h] = (kok && wok[r][h]) ? ld_stream(wrow[r][h] + k * 2) : zero;
#pragma unroll
        for (int m = 0; m < MT; ++m) st.x[m] = (kok && xok[m]) ? ld_cached(xrow[m] + k * 2) : zero;
    };
    auto compute = [&](const Step<RT, MT>& st) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // k-slots {2t,2t+1 | 2t+8,2t+9} <- this lane's k {0,1 | 2,3}, then {4,5 | 6,7}
                mma16816<kBf16>(acc[r][m], st.w[r][0].x, st.w[r][1].x, st.w[r][0].y,
                                st.w[r][1].y, st.x[m].x, st.x[m].y);
                mma16816<kBf16>(acc[r][m], st.w[r][0].z, st.w[r][1].z, st.w[r][0].w,
                                st.w[r][1].w, st.x[m].z, st.x[m].w);
            }
    };

    // Software pipeline: PF steps of loads in flight; ring slots are indexed
    // by compile-time constants so they stay in registers.
    Step<RT, MT> ring[PF];
#pragma unroll
    for (int u = 0; u < PF; ++u) load(ring[u], s_begin + u);
    for (int64_t s0 = s_begin; s0 < s_end; s0 += PF) {
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            if (s0 + u < s_end) {
                compute(ring[u]);
                load(ring[u], s0 + u + PF);
            }
        }
    }

    // D fragment: (row g, cols 2t, 2t+1) and (row g+8, same cols); rows are
    // weight rows (output columns n), columns are activation rows (m).
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            red[warp][r * 16 + g][m * 8 + 2 * t] = acc[r][m][0];
            red[warp][r * 16 + g][m * 8 + 2 * t + 1] = acc[r][m][1];
            red[warp][r * 16 + g + 8][m * 8 + 2 * t] = acc[r][m][2];
            red[warp][r * 16 + g + 8][m * 8 + 2 * t + 1] = acc[r][m][3];
        }
    __syncthreads();

    TOut* Y = static_cast<TOut*>(p.Y);
    for (int e = threadIdx.x; e < RT * 16 * MT * 8; e += WARPS * 32) {
        const int nl = e % (RT * 16), m = e / (RT * 16);  // consecutive threads: consecutive n
        const int64_t n = n0 + nl;
        if (m >= p.M || n >= p.N) continue;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) sum += red[w][nl][m];
        TOut* dst = Y + m * p.ldy + n;
        const float old = p.beta != 0.0f ? OutT<TOut>::load(dst) : 0.0f;
        OutT<TOut>::store(dst, axpby(p.alpha, sum, p.beta, old));
    }
}

// Chosen shape (measured on GB300 at N = K = 8192): 32 weight rows per CTA,
// 8 warps splitting K, 4 K-steps of loads in flight for M <= 8 and 3 for
// M <= 16 (where a deeper pipeline no longer fits the register budget).
constexpr int kRT = 2, kWarps = 8, kPF1 = 4, kPF2 = 3;

template <bool kBf16, typename TOut>
cudaError_t launch_typed(const Params& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.N + kRT * 16 - 1) / (kRT * 16)));
    if (p.M <= 8) skinny_kernel<kBf16, 1, TOut, kRT, kWarps, kPF1><<<grid, kWarps * 32, 0, s>>>(p);
    else skinny_kernel<kBf16, 2, TOut, kRT, kWarps, kPF2><<<grid, kWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool skinny_supports(const GemmArgs& a) {
    const bool types = (a.in_dtype == DGA_BF16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_BF16)) ||
                       (a.in_dtype == DGA_F16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_F16));
    return types && a.layout_b == DGA_COL_MAJOR && a.M >= 1 && a.M <= 16 && a.K % 8 == 0 &&
           a.lda % 8 == 0 && a.ldb % 8 == 0 && aligned(a.A, 16) && aligned(a.B, 16) &&
           (a.N + kRT * 16 - 1) / (kRT * 16) <= 0x7fffffff;
}

cudaError_t skinny_launch(const GemmArgs& a, int* launches) {
    Params p{a.M, a.N, a.K, a.A, a.lda, a.B, a.ldb, a.C, a.ldc, a.alpha_f, a.beta_f};
    cudaError_t e = cudaErrorInvalidValue;
    const bool bf = a.in_dtype == DGA_BF16;
    if (a.out_dtype == DGA_F32) e = bf ? launch_typed<true, float>(p, a.stream) : launch_typed<false, float>(p, a.stream);
    else if (a.out_dtype == DGA_BF16) e = launch_typed<true, __nv_bfloat16>(p, a.stream);
    else if (a.out_dtype == DGA_F16) e = launch_typed<false, __half>(p, a.stream);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace dga
