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
// once, in the access pattern HBM serves best, with enough bytes in flight,
// and (2) keep the arithmetic off the critical path.
//
//  * Streaming: each CTA owns a contiguous block of at most 64 weight rows and
//    walks K in stages of 256.  The grid is a whole number of waves of SMs
//    and the rows are shared out evenly (8192 rows on 152 SMs: 53 or 54 rows
//    per CTA), so every SM streams the same number of bytes; rows past a
//    CTA's share are zero-filled in shared memory and never read from HBM.  Every cp.async of a warp
//    copies 512 contiguous bytes of one row (16 bytes per lane, 256-byte L2
//    prefetch size) into a shared-memory ring of kStages stages; on GB300
//    this pattern streams a single pass over 128 MB at ~96% of the measured
//    copy bandwidth, where per-lane row-strided loads reach ~84%.  The M <= 16
//    activation rows of the same K range ride along in the same stage.
//  * Arithmetic: weight rows are the "A" operand and activation rows the "B"
//    operand of mma.sync m16n8k16 (fp32 accumulate), so a warp computes 16
//    weight rows x 8 activation rows per instruction, with fragments read by
//    ldmatrix from rows padded by 16 bytes (no bank conflicts).  The FP32
//    FMA pipe alone could not keep up at M = 16 (2 M FLOP per weight element
//    at ~7 TB/s is ~110 TFLOP/s).
//  * The 16 k-steps of a stage are spread over the 8 warps; at the end the
//    warps' partial tiles are summed in shared memory and the fused
//    alpha/beta epilogue writes Y.  Each CTA starts its walk over K at a
//    different stage, so the CTAs do not all read the same activation lines
//    at the same moment.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "dga_internal.h"
#include "epilogue.cuh"

namespace dga {
namespace {

constexpr int kWarps = 8;
constexpr int kKStage = 256;       // K per pipeline stage
constexpr int kStageCount = 4;     // stages in the shared-memory ring
constexpr int kRowBytes = kKStage * 2 + 16;  // padded shared-memory row (528 bytes)

struct Params {
    int64_t M, N, K;
    const void* X;
    int64_t ldx;
    const void* W;
    int64_t ldw;
    void* Y;
    int64_t ldy;
    float alpha, beta;
    const void* bias;  // N output-type values added to every row, or null
    int64_t ctas;      // grid size: CTA c owns rows [c*N/ctas, (c+1)*N/ctas)
};

// 16-byte async copy with zero fill: src_bytes (0 or 16) bytes are read, the
// rest of the 16 written as zeros.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    asm volatile(
        "cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(
            static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
        "l"(gmem), "r"(src_bytes)
        : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], const void* smem) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))));
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (kBf16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Shared memory: kStages x (kRows weight rows + 8*MT activation rows) padded
// rows.  The cross-warp reduction reuses the ring once the pipeline drains,
// keeping the footprint at two CTAs per SM.
template <int MT, int kRows>
struct SkinnySmem {
    static constexpr int kStages = kStageCount;
    static constexpr int kXRows = 8 * MT;
    static constexpr int kStageBytes = (kRows + kXRows) * kRowBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kRedBytes = kWarps * kRows * (MT * 8 + 1) * 4;
    static_assert(kRedBytes <= kRingBytes, "the reduction area lives in the ring");
    static constexpr int kTotal = kRingBytes;
};

// MT = number of 8-row activation tiles (1 for M <= 8, 2 for M <= 16);
// kRows = weight rows per CTA (a multiple of 16).
template <bool kBf16, int MT, int kRows, typename TOut>
__global__ void __launch_bounds__(kWarps * 32) skinny_kernel(Params p) {
    using S = SkinnySmem<MT, kRows>;
    constexpr int RT = kRows / 16;
    constexpr int kStages = S::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * p.N / p.ctas;
    const int64_t n_end = (static_cast<int64_t>(blockIdx.x) + 1) * p.N / p.ctas;  // n_end - n0 <= kRows
    const int64_t n_stages = (p.K + kKStage - 1) / kKStage;
    const char* W = static_cast<const char*>(p.W);
    const char* X = static_cast<const char*>(p.X);

    // Stage s: weight rows n0 .. n_end-1 and activation rows 0 .. 8*MT-1, k in
    // [s*256, s*256 + 256).  Chunk c of 16 bytes: row c / 32, column c % 32;
    // a warp's 32 lanes copy one row's 512 contiguous bytes.
    // CTAs start their walk over K at different stages, so that at any moment
    // they read different activation lines (all of them reading the same
    // lines at once makes those L2 lines a hot spot).  The order is fixed per
    // CTA, so results stay deterministic.
    const int64_t k_start = static_cast<int64_t>(blockIdx.x) % n_stages;
    auto load_stage = [&](int64_t s, int slot) {
        uint8_t* base = smem + slot * S::kStageBytes;
        int64_t ks = s + k_start;
        if (ks >= n_stages) ks -= n_stages;
        const int64_t k0 = ks * kKStage;
#pragma unroll
        for (int i = 0; i < (kRows + S::kXRows) * 32 / (kWarps * 32); ++i) {
            const int c = i * kWarps * 32 + tid;
            const int row = c >> 5, col = c & 31;
            const int64_t k = k0 + col * 8;
            const bool kok = k < p.K;  // K % 8 == 0: a chunk is wholly in or out
            const char* src;
            bool ok;
            if (row < kRows) {
                const int64_t n = n0 + row;
                ok = kok && n < n_end;
                src = W + ((ok ? n : 0) * p.ldw + (ok ? k : 0)) * 2;
            } else {
                const int64_t m = row - kRows;
                ok = kok && m < p.M;
                src = X + ((ok ? m : 0) * p.ldx + (ok ? k : 0)) * 2;
            }
            cp_async16(base + row * kRowBytes + col * 16, src, ok ? 16 : 0);
        }
    };

    float acc[RT][MT][4];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][m][i] = 0.0f;

    // ldmatrix row addresses: A (16 x 16 tile) lane -> row lane%16, k half lane/16;
    // B (8 activation rows x 16 k) lane -> row lane%8, k half (lane/8)%2.
    const int a_row = lane & 15, a_kh = lane >> 4;
    const int b_row = lane & 7, b_kh = (lane >> 3) & 1;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < n_stages) load_stage(s, s);
        cp_async_commit();
    }
    for (int64_t s = 0; s < n_stages; ++s) {
        cp_async_wait<kStages - 2>();  // stage s has landed (for this thread's copies)
        __syncthreads();               // ... and for everyone's; slot (s-1) is free
        const int64_t next = s + kStages - 1;
        if (next < n_stages) load_stage(next, static_cast<int>(next % kStages));
        cp_async_commit();

        const uint8_t* base = smem + static_cast<int>(s % kStages) * S::kStageBytes;
        const uint8_t* xbase = base + kRows * kRowBytes;
#pragma unroll
        for (int j = 0; j < kKStage / 16 / kWarps; ++j) {
            const int kk = (warp * (kKStage / 16 / kWarps) + j) * 16;  // k offset in the stage
            uint32_t a[RT][4];
#pragma unroll
            for (int r = 0; r < RT; ++r)
                ldmatrix_x4(a[r], base + (r * 16 + a_row) * kRowBytes + (kk + a_kh * 8) * 2);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint32_t b[2];
                ldmatrix_x2(b, xbase + (m * 8 + b_row) * kRowBytes + (kk + b_kh * 8) * 2);
#pragma unroll
                for (int r = 0; r < RT; ++r) mma16816<kBf16>(acc[r][m], a[r], b[0], b[1]);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring before it becomes `red`

    // D fragment: (row g, cols 2t, 2t+1) and (row g+8, same cols); rows are
    // weight rows (output columns n), columns are activation rows (m).
    float (*red)[kRows][MT * 8 + 1] = reinterpret_cast<float (*)[kRows][MT * 8 + 1]>(smem);
    const int g = lane >> 2, t = lane & 3;
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
    for (int e = tid; e < kRows * MT * 8; e += kWarps * 32) {
        const int nl = e % kRows, m = e / kRows;  // consecutive threads: consecutive n
        const int64_t n = n0 + nl;
        if (m >= p.M || n >= n_end) continue;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[w][nl][m];
        TOut* dst = Y + m * p.ldy + n;
        const float old = p.beta != 0.0f ? OutT<TOut>::load(dst) : 0.0f;
        float v = axpby(p.alpha, sum, p.beta, old);
        if (p.bias) v += OutT<TOut>::load(static_cast<const TOut*>(p.bias) + n);
        OutT<TOut>::store(dst, v);
    }
}

template <bool kBf16, int MT, int kRows, typename TOut>
cudaError_t launch_mt(const Params& p, cudaStream_t s) {
    auto kern = skinny_kernel<kBf16, MT, kRows, TOut>;
    const int smem = SkinnySmem<MT, kRows>::kTotal;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(static_cast<unsigned>(p.ctas)), kWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

// Weight rows per CTA, at most.  Each CTA also streams the activation rows of
// its K range, so activation bytes are (M / rows) of the weight bytes; blocks
// of up to 64 rows (one CTA per SM) measured fastest on GB300 for every
// M <= 16, e.g. M = 16: 5.06 TB/s with 64 rows against 4.46 TB/s with 32.
constexpr int kRowsPerCta = 64;

// CTAs: whole waves of one CTA per SM, as few as hold every row at <= 64 rows
// per CTA, but no more CTAs than 16-row tiles.
int64_t skinny_ctas(int64_t N, int sm_count) {
    const int64_t sms = sm_count > 0 ? sm_count : 1;
    const int64_t min_ctas = (N + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t waves = (min_ctas + sms - 1) / sms;
    return std::max<int64_t>(1, std::min(waves * sms, (N + 15) / 16));
}

template <bool kBf16, typename TOut>
cudaError_t launch_typed(const Params& p, cudaStream_t s) {
    return p.M <= 8 ? launch_mt<kBf16, 1, kRowsPerCta, TOut>(p, s)
                    : launch_mt<kBf16, 2, kRowsPerCta, TOut>(p, s);
}

}  // namespace

bool skinny_supports(const GemmArgs& a) {
    const bool types = (a.in_dtype == DGA_BF16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_BF16)) ||
                       (a.in_dtype == DGA_F16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_F16));
    return types && a.layout_a == DGA_ROW_MAJOR && a.layout_b == DGA_COL_MAJOR && a.M >= 1 &&
           a.M <= 16 && a.K % 8 == 0 &&
           a.lda % 8 == 0 && a.ldb % 8 == 0 && aligned(a.A, 16) && aligned(a.B, 16) &&
           (a.N + 15) / 16 <= 0x7fffffff;
}

cudaError_t skinny_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches) {
    Params p{a.M, a.N, a.K, a.A, a.lda, a.B, a.ldb, a.C, a.ldc, a.alpha_f, a.beta_f, a.bias,
             skinny_ctas(a.N, dev.sm_count)};
    if (p.ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaErrorInvalidValue;
    const bool bf = a.in_dtype == DGA_BF16;
    if (a.out_dtype == DGA_F32) e = bf ? launch_typed<true, float>(p, a.stream) : launch_typed<false, float>(p, a.stream);
    else if (a.out_dtype == DGA_BF16) e = launch_typed<true, __nv_bfloat16>(p, a.stream);
    else if (a.out_dtype == DGA_F16) e = launch_typed<false, __half>(p, a.stream);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace dga
