// sgemm_simt.cu -- exact FP32 GEMM on the SIMT FMA pipes (FFMA, never TF32).
//
// Design (the register-tiled kernel that "Matrix multiplication: arithmetic
// intensity, tiling and Tensor Core" sections 5.3-5.4 describe without code):
//   * a 128 x 128 block tile: every A and B element brought on chip is reused
//     128 times, so the DRAM-side intensity reaches ~32 FLOP/B (section 5.3:
//     I_tile = T/4), and the 129 MB L2 serves most re-reads;
//   * 256 threads, each accumulating an 8 x 8 register tile: per k, 8 A and 8
//     B values from shared memory feed 64 FFMAs (section 5.4: 4 FMA per
//     shared read);
//   * double buffering (section 5.4): the next K-slice is fetched from global
//     memory into registers with 128-bit loads while the current slice is
//     consumed, then written to the other shared-memory buffer, so one
//     barrier per slice suffices and load latency hides behind 512 FFMAs;
//   * A is stored k-major in shared memory (transposed on the way in) with
//     rows padded by 4 floats, so the transposing stores are free of bank
//     conflicts and the 8 A values per k are two 128-bit broadcast loads
//     (the padding remedy of section 5.7);
//   * edges: loads outside M, N or K return zero, stores are masked.
//
// Thread layout: 8 warps tile the block as 2 (M) x 4 (N) warp tiles of
// 64 x 32; inside a warp, lane = lm * 4 + ln with lm in 0..7, ln in 0..3.  A
// thread owns rows {wm*64 + lm*4 + i, wm*64 + 32 + lm*4 + i} and columns
// {wn*32 + ln*4 + j, wn*32 + 16 + ln*4 + j}, i, j in 0..3.
#include "dga_internal.h"
#include "epilogue.cuh"

namespace dga {
namespace {

constexpr int BM = 128, BN = 128, BK = 8;
constexpr int kThreads = 256;
constexpr int kApad = 4;  // floats of padding per k-row of the transposed A tile

struct Params {
    int64_t M, N, K;
    const float* A;
    int64_t lda;
    const float* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
    float alpha, beta;
    int vec_c;  // C is 16-byte aligned and ldc % 4 == 0: float4 epilogue
    int vec_a;  // A 16-byte aligned and lda % 4 == 0: float4 loads of A
    int vec_b;  // the same for B
};

__device__ __forceinline__ float4 ld_f4_masked(const float* row, int64_t col, int64_t ncols,
                                               bool row_ok, bool vec) {
    if (vec && row_ok && col + 3 < ncols) return __ldg(reinterpret_cast<const float4*>(row + col));
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (row_ok && col + i < ncols) ? __ldg(row + col + i) : 0.0f;
    return make_float4(v[0], v[1], v[2], v[3]);
}

__global__ void __launch_bounds__(kThreads, 2) sgemm_128x128_kernel(Params p) {
    __shared__ __align__(16) float As[2][BK][BM + kApad];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;
    const int lm = lane >> 2, ln = lane & 3;
    const int64_t row0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t col0 = static_cast<int64_t>(blockIdx.x) * BN;

    // Global -> register staging: A tile 128 x 8 (thread: row tid/2, k 4*(tid%2)),
    // B tile 8 x 128 (thread: k tid/32, column 4*(tid%32)).
    const int a_r = tid >> 1, a_k = (tid & 1) * 4;
    const int b_k = tid >> 5, b_c = (tid & 31) * 4;
    const int64_t a_grow = row0 + a_r;
    const bool a_row_ok = a_grow < p.M;
    const float* a_src = p.A + (a_row_ok ? a_grow : 0) * p.lda;
    const int64_t b_gcol = col0 + b_c;

    const bool vec_a = p.vec_a != 0, vec_b = p.vec_b != 0;
    auto load_a = [&](int64_t k0) { return ld_f4_masked(a_src, k0 + a_k, p.K, a_row_ok, vec_a); };
    auto load_b = [&](int64_t k0) {
        int64_t gk = k0 + b_k;
        bool ok = gk < p.K;
        const float* row = p.B + (ok ? gk : 0) * p.ldb;
        return ld_f4_masked(row, b_gcol, p.N, ok, vec_b);
    };
    auto stash = [&](int buf, float4 a, float4 b) {
        As[buf][a_k + 0][a_r] = a.x;
        As[buf][a_k + 1][a_r] = a.y;
        As[buf][a_k + 2][a_r] = a.z;
        As[buf][a_k + 3][a_r] = a.w;
        *reinterpret_cast<float4*>(&Bs[buf][b_k][b_c]) = b;
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    const int am0 = wm * 64 + lm * 4, am1 = am0 + 32;
    const int bn0 = wn * 32 + ln * 4, bn1 = bn0 + 16;

    const int64_t n_slices = (p.K + BK - 1) / BK;
    if (n_slices > 0) {
        stash(0, load_a(0), load_b(0));
        __syncthreads();
    }
    for (int64_t s = 0; s < n_slices; ++s) {
        const int buf = static_cast<int>(s & 1);
        const bool more = s + 1 < n_slices;
        float4 na, nb;
        if (more) {
            na = load_a((s + 1) * BK);
            nb = load_b((s + 1) * BK);
        }
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
            *reinterpret_cast<float4*>(&a[0]) = *reinterpret_cast<const float4*>(&As[buf][k][am0]);
            *reinterpret_cast<float4*>(&a[4]) = *reinterpret_cast<const float4*>(&As[buf][k][am1]);
            *reinterpret_cast<float4*>(&b[0]) = *reinterpret_cast<const float4*>(&Bs[buf][k][bn0]);
            *reinterpret_cast<float4*>(&b[4]) = *reinterpret_cast<const float4*>(&Bs[buf][k][bn1]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
            // The other buffer was last read in slice s-1, and every thread
            // passed the barrier at the end of slice s-1 after that read.
            stash(buf ^ 1, na, nb);
        }
        __syncthreads();
    }

    // Epilogue: out = alpha*acc + beta*C, masked; float4 where aligned.
    const bool vec_ok = p.vec_c != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + (i < 4 ? am0 + i : am1 + (i - 4));
        if (r >= p.M) continue;
        float* crow = p.C + r * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t c = col0 + (h == 0 ? bn0 : bn1);
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = acc[i][h * 4 + j];
            if (vec_ok && c + 3 < p.N) {
                float4* dst = reinterpret_cast<float4*>(crow + c);
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.beta != 0.0f) o = *dst;
                o.x = axpby(p.alpha, v[0], p.beta, o.x);
                o.y = axpby(p.alpha, v[1], p.beta, o.y);
                o.z = axpby(p.alpha, v[2], p.beta, o.z);
                o.w = axpby(p.alpha, v[3], p.beta, o.w);
                *dst = o;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (c + j < p.N) {
                        float old = p.beta != 0.0f ? crow[c + j] : 0.0f;
                        crow[c + j] = axpby(p.alpha, v[j], p.beta, old);
                    }
                }
            }
        }
    }
}

}  // namespace

bool simt_supports(const GemmArgs& a) {
    return a.in_dtype == DGA_F32 && a.out_dtype == DGA_F32 && a.layout_b == DGA_ROW_MAJOR &&
           (a.M + BM - 1) / BM <= 65535;
}

cudaError_t simt_launch(const GemmArgs& a, int* launches) {
    Params p{a.M, a.N, a.K, static_cast<const float*>(a.A), a.lda,
             static_cast<const float*>(a.B), a.ldb, static_cast<float*>(a.C), a.ldc,
             a.alpha_f, a.beta_f, (a.ldc % 4 == 0 && aligned(a.C, 16)) ? 1 : 0,
             (a.lda % 4 == 0 && aligned(a.A, 16)) ? 1 : 0, (a.ldb % 4 == 0 && aligned(a.B, 16)) ? 1 : 0};
    dim3 grid(static_cast<unsigned>((a.N + BN - 1) / BN), static_cast<unsigned>((a.M + BM - 1) / BM));
    sgemm_128x128_kernel<<<grid, kThreads, 0, a.stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace dga
