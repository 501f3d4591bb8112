// sgemm_simt.cu -- exact FP32 GEMM on the SIMT FMA pipes (FFMA, never TF32).
//
// Design (the register-tiled kernel that "Matrix multiplication: arithmetic
// intensity, tiling and Tensor Core" sections 5.3-5.4 describe without code):
//   * a 128 x 128 block tile: every A and B element brought on chip is reused
//     128 times, so the DRAM-side intensity reaches ~32 FLOP/B (section 5.3:
//     I_tile = T/4), and the 129 MB L2 serves most re-reads;
//   * 256 threads, each accumulating an 8 x 8 register tile: per k, 8 A and 8
//     B values from shared memory feed 64 FMAs (section 5.4: 4 FMA per
//     shared read), issued as 32 packed fma.rn.f32x2 -- each half an
//     ordinary round-to-nearest fp32 FMA, so the results are those of 64
//     scalar FFMAs in the same order;
//   * double buffering (section 5.4) at two levels: the next K-slice (8 deep)
//     is fetched from global memory into registers with 128-bit loads while
//     the current slice is consumed, then written to the other shared-memory
//     buffer (one barrier per slice); and inside a slice the fragments of
//     k+1 are read from shared memory while the FMAs of k run.  A slice of
//     8 keeps the staging registers few enough for two CTAs per SM at 128
//     registers, which measured faster than deeper slices on GB300;
//   * A is stored k-major in shared memory (transposed on the way in); each
//     warp stages 32 consecutive rows at one k, so the transposing stores hit
//     32 consecutive words (no bank conflicts), and the 8 A values a thread
//     needs per k are two 128-bit broadcast loads;
//   * both operand layouts: a column-major A arrives k-major and is copied
//     with 128-bit stores, a column-major B (N x K, e.g. the W^T of a
//     fully-connected layer) takes the transposing stores of a row-major A;
//     the epilogue adds an optional bias row;
//   * tiles that lie wholly inside the matrices (and a K range that is a
//     whole number of slices) run a copy of the main loop without any bounds
//     checks; edge tiles load zeros outside M, N and K and mask their stores;
//   * problems with fewer tiles than resident blocks cut every tile along K
//     into 2-4 ranges whose partial sums go to the caller's workspace and are
//     added in a fixed order by a second small kernel, so that most SMs are
//     not left idle.
//
// Thread layout: 8 warps tile the block as 2 (M) x 4 (N) warp tiles of
// 64 x 32; inside a warp, lane = lm * 4 + ln with lm in 0..7, ln in 0..3.  A
// thread owns rows {wm*64 + lm*4 + i, wm*64 + 32 + lm*4 + i} and columns
// {wn*32 + ln*4 + j, wn*32 + 16 + ln*4 + j}, i, j in 0..3.
#include <algorithm>

#include "dga_internal.h"
#include "epilogue.cuh"

namespace dga {
namespace {

constexpr int BM = 128, BN = 128, BK = 8;
constexpr int kThreads = 256;
constexpr int kAStride = BM + 4;  // floats per k-row of the A and B tiles (BM == BN)
constexpr int64_t kSimtMaxK = int64_t{1} << 33;  // larger K: the generic kernel
constexpr int kSimtBlocksPerSm = 2;  // register budget: 65536 / (256 * 2) = 128 per thread

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
    // Tile schedule: tile t covers rows (t / tiles_n)*BM, columns (t % tiles_n)*BN.
    // Blocks below full_tiles own one tile each; each block above owns one of
    // `parts` K-ranges (part_k deep) of a tail tile and writes its partial
    // product to `partials` (BM x BN floats per block, row-major).
    int64_t tiles_n, full_tiles, part_k;
    int parts;
    float* partials;
    const float* bias;  // N values added to every row, or null
    // Wide kernel, stream-K schedule (sk_ctas > 0): the (tile, 16-deep
    // K-slice) units, sk_slices per tile, are cut into sk_ctas equal
    // contiguous ranges, one per block; see sgemm_wide_sk_kernel.
    int64_t sk_units, sk_slices;
    int sk_ctas;
};

struct Smem {
    float A[2][BK][kAStride];  // A[buf][k][m]
    float B[2][BK][kAStride];  // B[buf][k][n] (padded like A: see the staging roles)
};

__device__ __forceinline__ float4 ld_f4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

// Packed pairs of fp32 values in one 64-bit register: low half first.
__device__ __forceinline__ uint64_t pair_of(float v) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void unpair(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

// d.lo += a.lo * b.lo and d.hi += a.hi * b.hi, each one fp32 fused
// multiply-add rounded to nearest: two FFMAs' results in one instruction.
__device__ __forceinline__ void fma2(uint64_t& d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// Four consecutive elements of a row starting at `col`; zeros outside.
__device__ __forceinline__ float4 ld_f4_checked(const float* row, int64_t col, int64_t ncols,
                                                bool row_ok, bool vec) {
    if (vec && row_ok && col + 3 < ncols) return ld_f4(row + col);
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (row_ok && col + i < ncols) ? __ldg(row + col + i) : 0.0f;
    return make_float4(v[0], v[1], v[2], v[3]);
}

// One block tile over K in [k_begin, k_end).  kChecked = false only for
// tiles wholly inside M, N whose K range is a whole number of slices, with
// 16-byte-friendly A and B.  `partial` non-null: write the raw accumulators
// there (BM x BN, row-major) instead of the alpha/beta epilogue.
// kTransA: A is stored K x M (column-major A), so its K-slice arrives
// already k-major and is copied like row-major B, without the transposing
// stores.  kTransB: B is stored N x K (column-major B); its slice is staged
// the way row-major A is, through transposing stores.
// kRunPtr: interior slices walk A and B with running pointers instead of
// recomputing the addresses; measured faster for a column-major B (4096^3:
// 56.6 against 54.8 TFLOP/s, and 57.1 against 48.5 with a bias row) and no
// different otherwise, so the interior kernel uses it for column-major B.
// kColOuter: the order of the 32 packed FMAs of a k-step (see the loop); the
// interior kernel takes column pairs outer, the general kernel rows outer
// (the other order needs registers it does not have: it spilled there).
template <bool kChecked, bool kTransA, bool kTransB, int kReadC = -1, int kBias = -1,
          bool kRunPtr = false, bool kColOuter = false>
__device__ __forceinline__ void block_tile(const Params& p, Smem& sm, int64_t row0, int64_t col0,
                                           int64_t k_begin, int64_t k_end, float* partial) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // staging roles (one float4 of A and one of B per thread and slice):
    // row-major A: row 16*warp + lane/2 at k offset 4*(lane%2) -- a lane pair
    // reads one whole 32-byte sector of a row, and the transposing stores of
    // a warp (16 rows, k and k+4; the padded stride puts k+4 16 banks away)
    // hit 32 different banks; row-major B: row k = warp, columns 4*lane ..
    // 4*lane + 3.  Column-major A is staged like row-major B (k = warp, rows
    // 4*lane .. 4*lane + 3), column-major B like row-major A.  The lane-pair
    // sectors measured 5-10% faster on GB300 than one float4 per row per warp.
    const int a_k = kTransA ? warp : (lane & 1) * 4;
    const int a_r = kTransA ? lane * 4 : warp * 16 + (lane >> 1);
    const int b_k = kTransB ? (lane & 1) * 4 : warp;
    const int b_c = kTransB ? warp * 16 + (lane >> 1) : lane * 4;
    const bool a_ok = kTransA || !kChecked || row0 + a_r < p.M;
    const bool b_ok = !kTransB || !kChecked || col0 + b_c < p.N;
    const float* a_src = kTransA ? p.A + row0 + a_r : p.A + (a_ok ? row0 + a_r : 0) * p.lda;
    const float* b_src = kTransB ? p.B + (b_ok ? col0 + b_c : 0) * p.ldb : p.B + col0 + b_c;
    const bool vec_a = p.vec_a != 0, vec_b = p.vec_b != 0;
    const float* a_run = kTransA ? a_src + (k_begin + a_k) * p.lda : a_src + k_begin + a_k;
    const float* b_run = kTransB ? b_src + k_begin + b_k : b_src + (k_begin + b_k) * p.ldb;
    const int64_t a_step = kTransA ? BK * p.lda : BK;
    const int64_t b_step = kTransB ? BK : BK * p.ldb;

    float4 ra, rb;
    auto fetch = [&](int64_t k0) {
        if constexpr (!kChecked && kRunPtr) {
            ra = ld_f4(a_run);
            a_run += a_step;
            rb = ld_f4(b_run);
            b_run += b_step;
        } else if constexpr (!kChecked) {
            ra = kTransA ? ld_f4(a_src + (k0 + a_k) * p.lda) : ld_f4(a_src + k0 + a_k);
            rb = kTransB ? ld_f4(b_src + k0 + b_k) : ld_f4(b_src + (k0 + b_k) * p.ldb);
        } else {
            if constexpr (kTransA) {
                const bool kok = k0 + a_k < k_end;
                ra = ld_f4_checked(p.A + (kok ? k0 + a_k : 0) * p.lda, row0 + a_r, p.M, kok, vec_a);
            } else {
                ra = ld_f4_checked(a_src, k0 + a_k, k_end, a_ok, vec_a);
            }
            if constexpr (kTransB) {
                rb = ld_f4_checked(b_src, k0 + b_k, k_end, b_ok, vec_b);
            } else {
                const bool kok = k0 + b_k < k_end;
                rb = ld_f4_checked(p.B + (kok ? k0 + b_k : 0) * p.ldb, col0 + b_c, p.N, kok, vec_b);
            }
        }
    };
    auto stash = [&](int buf) {
        if constexpr (kTransA) {
            *reinterpret_cast<float4*>(&sm.A[buf][a_k][a_r]) = ra;
        } else {
            sm.A[buf][a_k + 0][a_r] = ra.x;
            sm.A[buf][a_k + 1][a_r] = ra.y;
            sm.A[buf][a_k + 2][a_r] = ra.z;
            sm.A[buf][a_k + 3][a_r] = ra.w;
        }
        if constexpr (kTransB) {
            sm.B[buf][b_k + 0][b_c] = rb.x;
            sm.B[buf][b_k + 1][b_c] = rb.y;
            sm.B[buf][b_k + 2][b_c] = rb.z;
            sm.B[buf][b_k + 3][b_c] = rb.w;
        } else {
            *reinterpret_cast<float4*>(&sm.B[buf][b_k][b_c]) = rb;
        }
    };

    // compute roles: 2 (M) x 4 (N) warp tiles of 64 x 32; lane = lm*4 + ln
    const int wm = warp >> 2, wn = warp & 3;
    const int lm = lane >> 2, ln = lane & 3;
    const int am0 = wm * 64 + lm * 4, am1 = am0 + 32;
    const int bn0 = wn * 32 + ln * 4, bn1 = bn0 + 16;

    // accumulators as pairs of adjacent columns: acc2[i][q] holds columns
    // 2q and 2q+1 of row i, updated by one fma.rn.f32x2 (two independent
    // IEEE fp32 fused multiply-adds: the same results as two fmaf)
    uint64_t acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc2[i][q] = 0ull;  // (+0.0f, +0.0f)

    // slices counted in 32 bits (simt_supports keeps K below 2^33): a 64-bit
    // counter measured 1.5-5% slower in the wide kernel's main loop; here the
    // same on average (58.0 against 57.8 TFLOP/s over the eight layout and
    // epilogue variants at 4096^3)
    const int n_slices = static_cast<int>((k_end - k_begin + BK - 1) / BK);
    fetch(k_begin);
    stash(0);
    __syncthreads();
    for (int s = 0; s < n_slices; ++s) {
        const int buf = static_cast<int>(s & 1);
        const bool more = s + 1 < n_slices;
        // Fragments are double-buffered in registers: the shared-memory loads
        // for k+1 are issued before the 64 FMAs of k.  The next slice's global
        // loads go out after two k-steps (their registers are live for less of
        // the loop; 4096^3 measured 56.0 -> 57.7 TFLOP/s on GB300, any fetch
        // point from k = 1 to 4 the same).  The 64 FMAs of a k-step are 32
        // packed fma.rn.f32x2 on column pairs, each a_i broadcast into both
        // halves: half the issue slots of scalar FFMAs.  Measured at 4096^3
        // over the four operand layouts, with beta or a bias row (mean /
        // lowest of the eight, TFLOP/s): scalar FFMAs 57.1 / 52.4, packed
        // with rows outer 57.6 / 54.9, packed with column pairs outer (the 8
        // broadcasts made first) 57.9 / 55.4.  Keeping A as ready-made
        // (a, a) pairs in shared memory instead measured 50.1 (twice the A
        // bytes through the shared-memory pipe).
        float a[2][8];
        uint64_t b[2][4];  // column pairs (2q, 2q+1) of this thread's 8 B values
        auto frag = [&](int d, int k) {
            *reinterpret_cast<float4*>(&a[d][0]) = *reinterpret_cast<const float4*>(&sm.A[buf][k][am0]);
            *reinterpret_cast<float4*>(&a[d][4]) = *reinterpret_cast<const float4*>(&sm.A[buf][k][am1]);
            *reinterpret_cast<ulonglong2*>(&b[d][0]) = *reinterpret_cast<const ulonglong2*>(&sm.B[buf][k][bn0]);
            *reinterpret_cast<ulonglong2*>(&b[d][2]) = *reinterpret_cast<const ulonglong2*>(&sm.B[buf][k][bn1]);
        };
        frag(0, 0);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            if (k == 2 && more) fetch(k_begin + static_cast<int64_t>(s + 1) * BK);
            if (k + 1 < BK) frag((k + 1) & 1, k + 1);
            if constexpr (kColOuter) {
                uint64_t ap[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ap[i] = pair_of(a[k & 1][i]);  // (a_i, a_i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 8; ++i) fma2(acc2[i][q], ap[i], b[k & 1][q]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t ai = pair_of(a[k & 1][i]);  // (a_i, a_i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) fma2(acc2[i][q], ai, b[k & 1][q]);
                }
            }
        }
        // The other buffer was last read in slice s-1, before the barrier
        // that ended it, so it can be overwritten now.
        if (more) stash(buf ^ 1);
        __syncthreads();
    }

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) unpair(acc2[i][q], acc[i][2 * q], acc[i][2 * q + 1]);

    if (partial != nullptr) {
        // a K-range of a tail tile: raw partial sums, reduced by sgemm_tail_reduce
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float* prow = partial + (i < 4 ? am0 + i : am1 + (i - 4)) * BN;
            *reinterpret_cast<float4*>(prow + bn0) = *reinterpret_cast<const float4*>(&acc[i][0]);
            *reinterpret_cast<float4*>(prow + bn1) = *reinterpret_cast<const float4*>(&acc[i][4]);
        }
        return;
    }

    // Epilogue: out = alpha*acc + beta*C, float4 where aligned, masked at edges.
    // kReadC: 1 / 0 when the caller already knows whether beta != 0 (and
    // that C takes float4 stores), -1 to decide at run time.
    const bool vec_c = kReadC >= 0 || p.vec_c != 0;
    const bool read_c = kReadC >= 0 ? kReadC == 1 : p.beta != 0.0f;
    // the bias row (fully-connected layer): this thread's 8 columns, once.
    // kBias: 1 / 0 when the caller knows whether there is one (the kernel
    // without it then keeps the register allocation of a plain GEMM, which
    // measured 5% faster at 4096^3 than a run-time test), -1 to test here.
    const bool has_bias = kBias >= 0 ? kBias == 1 : p.bias != nullptr;
    float bv[8];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = col0 + (h == 0 ? bn0 : bn1) + j;
            bv[h * 4 + j] = (has_bias && (!kChecked || c < p.N)) ? p.bias[c] : 0.0f;
        }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + (i < 4 ? am0 + i : am1 + (i - 4));
        if (kChecked && r >= p.M) continue;
        float* crow = p.C + r * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t c = col0 + (h == 0 ? bn0 : bn1);
            const float* v = &acc[i][h * 4];
            if (vec_c && (!kChecked || c + 3 < p.N)) {
                float4* dst = reinterpret_cast<float4*>(crow + c);
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (read_c) o = *dst;
                o.x = axpby(p.alpha, v[0], p.beta, o.x);
                o.y = axpby(p.alpha, v[1], p.beta, o.y);
                o.z = axpby(p.alpha, v[2], p.beta, o.z);
                o.w = axpby(p.alpha, v[3], p.beta, o.w);
                if (has_bias) {  // (x + 0 is not x for x = -0, so no add without a bias)
                    o.x += bv[h * 4 + 0];
                    o.y += bv[h * 4 + 1];
                    o.z += bv[h * 4 + 2];
                    o.w += bv[h * 4 + 3];
                }
                *dst = o;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!kChecked || c + j < p.N) {
                        const float old = read_c ? crow[c + j] : 0.0f;
                        const float o = axpby(p.alpha, v[j], p.beta, old);
                        crow[c + j] = has_bias ? o + bv[h * 4 + j] : o;
                    }
                }
            }
        }
    }
}

// Tile order: groups of kGroupRows tile rows, walked column by column, so
// that the blocks resident at one time share A and B panels in L2 (measured
// 7% faster than row-by-row order at 4096^3 on GB300).
constexpr int kGroupRows = 8;

__device__ __forceinline__ void grouped_tile(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                             int64_t& tm, int64_t& tn) {
    const int64_t group_size = kGroupRows * tiles_n;
    const int64_t first = (t / group_size) * kGroupRows;
    const int64_t rows = min(tiles_m - first, static_cast<int64_t>(kGroupRows));
    const int64_t r = t % group_size;
    tm = first + r % rows;
    tn = r / rows;
}

// The general kernel: any shape, edge tiles, optional K split (1-D grid over
// the tile schedule).
template <int kMinBlocks, bool kTransA, bool kTransB>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sgemm_128x128_kernel(Params p) {
    __shared__ __align__(16) Smem sm;
    const int64_t b = blockIdx.x;
    int64_t tile, k_begin = 0, k_end = p.K;
    float* partial = nullptr;
    if (b < p.full_tiles) {
        tile = b;
    } else {
        const int64_t u = b - p.full_tiles;
        tile = p.full_tiles + u / p.parts;
        k_begin = (u % p.parts) * p.part_k;
        k_end = min(p.K, k_begin + p.part_k);
        partial = p.partials + u * (BM * BN);
    }
    int64_t tm, tn;
    grouped_tile(tile, (p.M + BM - 1) / BM, p.tiles_n, tm, tn);
    const int64_t row0 = tm * BM;
    const int64_t col0 = tn * BN;
    const bool interior = row0 + BM <= p.M && col0 + BN <= p.N && (k_end - k_begin) % BK == 0 &&
                          p.vec_a && p.vec_b;
    if (interior) block_tile<false, kTransA, kTransB, -1, -1, kTransB>(p, sm, row0, col0, k_begin, k_end, partial);
    else block_tile<true, kTransA, kTransB>(p, sm, row0, col0, k_begin, k_end, partial);
}

// The same tile code, specialised for problems made only of interior tiles
// (M, N multiples of 128, K of 8, 16-byte-friendly A, B and C) with no K
// split: one code path, a 2-D grid and the C read decided at compile time,
// which measured faster on GB300 than the general kernel at 4096^3.
template <int kMinBlocks, bool kTransA, bool kTransB, int kReadC, int kBias>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sgemm_128x128_interior_kernel(Params p) {
    __shared__ __align__(16) Smem sm;
    int64_t tm, tn;
    grouped_tile(static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x, gridDim.y, gridDim.x,
                 tm, tn);
    block_tile<false, kTransA, kTransB, kReadC, kBias, kTransB, true>(p, sm, tm * BM, tn * BN,
                                                                      0, p.K, nullptr);
}

// Sums the K-range partials of each tail tile in part order (so the result
// does not depend on which block finished first) and applies the epilogue.
// kTailSlabs blocks share a tile, 8 rows each (one float4 per thread), so
// that enough loads are in flight to keep this short step bandwidth-bound.
constexpr int kTailSlabs = BM / 8;

__global__ void __launch_bounds__(kThreads) sgemm_tail_reduce(Params p) {
    const int64_t slot = blockIdx.x / kTailSlabs;
    const int slab = static_cast<int>(blockIdx.x % kTailSlabs);
    const int64_t tile = p.full_tiles + slot;
    int64_t tm, tn;
    grouped_tile(tile, (p.M + BM - 1) / BM, p.tiles_n, tm, tn);
    const int64_t row0 = tm * BM;
    const int64_t col0 = tn * BN;
    const float* base = p.partials + slot * p.parts * (BM * BN);
    {
        const int e = slab * (8 * BN / 4) + threadIdx.x;
        const int r = e / (BN / 4), c = (e % (BN / 4)) * 4;
        float4 sum = *reinterpret_cast<const float4*>(base + r * BN + c);
        for (int q = 1; q < p.parts; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(base + q * (BM * BN) + r * BN + c);
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
        }
        const int64_t row = row0 + r, col = col0 + c;
        if (row >= p.M) return;
        float* crow = p.C + row * p.ldc;
        const float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (col + j < p.N) {
                const float old = p.beta != 0.0f ? crow[col + j] : 0.0f;
                const float o = axpby(p.alpha, v[j], p.beta, old);
                crow[col + j] = p.bias ? o + p.bias[col + j] : o;
            }
        }
    }
}

// How the tiles are scheduled.  With at least one full wave of tiles, whole
// tiles only: a block alone on its SM in the last, partial wave runs faster
// than paired blocks do, and splitting that wave along K measured slower at
// 4096^3 on GB300.  With fewer tiles than resident blocks, most SMs would
// idle, so every tile is cut along K into `parts` ranges (2-4, each at least
// 256 deep) whose partial sums are added afterwards.  parts == 1: no split.
struct Schedule {
    int64_t tiles, tiles_n, full_tiles, part_k;
    int parts;
    size_t partial_bytes;
};

Schedule plan_schedule(int64_t M, int64_t N, int64_t K, int sm_count) {
    Schedule sc{};
    sc.tiles_n = (N + BN - 1) / BN;
    sc.tiles = ((M + BM - 1) / BM) * sc.tiles_n;
    sc.full_tiles = sc.tiles;
    sc.parts = 1;
    sc.part_k = K;
    const int64_t slots = static_cast<int64_t>(kSimtBlocksPerSm) * sm_count;
    if (slots <= 0 || sc.tiles >= slots) return sc;
    const int64_t tail = sc.tiles;
    int64_t parts = std::min<int64_t>(4, slots / tail);
    parts = std::min<int64_t>(parts, K / 256);  // keep every part at least 256 deep
    if (parts < 2) return sc;
    const int64_t part_k = ((K + parts - 1) / parts + BK - 1) / BK * BK;
    parts = (K + part_k - 1) / part_k;
    if (parts < 2) return sc;
    sc.full_tiles = sc.tiles - tail;
    sc.parts = static_cast<int>(parts);
    sc.part_k = part_k;
    sc.partial_bytes = static_cast<size_t>(tail) * parts * BM * BN * sizeof(float);
    return sc;
}

// ---- the wide kernel: 128 x 256 block tiles, 8 x 16 per thread --------------
//
// For problems made of whole 128 x 256 tiles with at least one full wave of
// them, one block per SM holding twice the accumulators of the 128 x 128
// kernel does more FMAs per shared-memory read and per broadcast (per k, 8 A
// and 16 B values feed 128 FMAs: 64 packed fma.rn.f32x2 behind 8 pair
// broadcasts and 6 128-bit shared loads), and its 16-deep K slices halve the
// barriers per FMA.  It uses up to 255 registers, so one block of 8 warps per
// SM.  Measured on GB300 at whole waves (M = 4864, N = K = 4096): 64.6
// TFLOP/s against 60.6 for two 128 x 128 blocks per SM (66.8 once the slice
// loop counted in 32 bits).  With one block per SM a part-filled last wave
// would leave SMs idle for a whole tile time, so problems that are not a
// whole number of waves run the whole waves tile by tile and the rest on a
// stream-K schedule (sgemm_wide_sk_kernel): every block does the same share
// of the remaining (tile, K-slice) work, and the tiles split between blocks
// are summed in a fixed order by sgemm_wide_sk_reduce.  Thread layout: 8
// warps as 2 (M) x 4 (N)
// warp tiles of 64 x 64; lane = lm * 4 + ln; a thread owns rows {wm*64 +
// lm*4 + i, wm*64 + 32 + lm*4 + i} and columns {wn*64 + h*16 + ln*4 + j},
// i, j in 0..3, h in 0..3.  The results equal the 128 x 128 kernel's bit for
// bit (the same FMAs per element in the same k order).

constexpr int kWBM = 128, kWBN = 256, kWBK = 16;
constexpr int kWAStride = kWBM + 4;  // floats per k-row of the A tile
// and of the B tile: padded for a column-major B (keeps its transposing
// stores free of bank conflicts), unpadded for a row-major one (whose stores
// and reads each stay within one k-row)
template <bool kTransB>
struct WideSmem {
    static constexpr int kBStride = kWBN + (kTransB ? 4 : 0);
    float A[2][kWBK][kWAStride];
    float B[2][kWBK][kBStride];
};

__device__ __forceinline__ void wide_tile(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                          int64_t& tm, int64_t& tn) {
    grouped_tile(t, tiles_m, tiles_n, tm, tn);
}

// One 128 x 256 tile over K in [k_begin, k_end) (a whole number of slices,
// every element inside the matrices).  partial non-null: the raw
// accumulators go there (128 x 256 floats, row-major) instead of the
// epilogue.
template <bool kTransA, bool kTransB, int kReadC, int kBias>
__device__ __forceinline__ void wide_block_tile(const Params& p, WideSmem<kTransB>& sm, int64_t row0,
                                                int64_t col0, int64_t k_begin, int64_t k_end,
                                                float* partial) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // Staging roles per 16-deep slice (2 float4 of A and 4 of B per thread):
    //  row-major A: row 16*warp + lane/2, k 4*(lane%2) + 8v (v = 0, 1): a lane
    //    pair reads a whole 32-byte sector; transposing stores, conflict-free;
    //  column-major A (stored K x M): k = warp + 8v, rows 4*lane .. 4*lane+3;
    //  row-major B: k = warp + 8v, columns 4*lane + 128u (u = 0, 1);
    //  column-major B (stored N x K): column 16*warp + lane/2 + 128u, k
    //    4*(lane%2) + 8v, staged like row-major A.
    const float* a_run;
    const float* b_run;
    if constexpr (kTransA) a_run = p.A + (k_begin + warp) * p.lda + row0 + lane * 4;
    else a_run = p.A + (row0 + warp * 16 + (lane >> 1)) * p.lda + k_begin + (lane & 1) * 4;
    if constexpr (kTransB) b_run = p.B + (col0 + warp * 16 + (lane >> 1)) * p.ldb + k_begin + (lane & 1) * 4;
    else b_run = p.B + (k_begin + warp) * p.ldb + col0 + lane * 4;
    const int64_t a_step = kTransA ? kWBK * p.lda : kWBK;
    const int64_t b_step = kTransB ? kWBK : kWBK * p.ldb;
    float4 ra[2], rb[4];
    auto fetch = [&]() {
#pragma unroll
        for (int v = 0; v < 2; ++v) ra[v] = ld_f4(a_run + (kTransA ? 8 * v * p.lda : 8 * v));
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int v = 0; v < 2; ++v)
                rb[u * 2 + v] = kTransB ? ld_f4(b_run + 128 * u * p.ldb + 8 * v)
                                        : ld_f4(b_run + 8 * v * p.ldb + 128 * u);
        a_run += a_step;
        b_run += b_step;
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            if constexpr (kTransA) {
                *reinterpret_cast<float4*>(&sm.A[buf][warp + 8 * v][lane * 4]) = ra[v];
            } else {
                const int k = (lane & 1) * 4 + 8 * v, r = warp * 16 + (lane >> 1);
                sm.A[buf][k + 0][r] = ra[v].x;
                sm.A[buf][k + 1][r] = ra[v].y;
                sm.A[buf][k + 2][r] = ra[v].z;
                sm.A[buf][k + 3][r] = ra[v].w;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const float4 x = rb[u * 2 + v];
                if constexpr (kTransB) {
                    const int k = (lane & 1) * 4 + 8 * v, c = warp * 16 + (lane >> 1) + 128 * u;
                    sm.B[buf][k + 0][c] = x.x;
                    sm.B[buf][k + 1][c] = x.y;
                    sm.B[buf][k + 2][c] = x.z;
                    sm.B[buf][k + 3][c] = x.w;
                } else {
                    *reinterpret_cast<float4*>(&sm.B[buf][warp + 8 * v][lane * 4 + 128 * u]) = x;
                }
            }
    };

    const int wm = warp >> 2, wn = warp & 3;
    const int lm = lane >> 2, ln = lane & 3;
    const int am0 = wm * 64 + lm * 4, am1 = am0 + 32;
    const int bn0 = wn * 64 + ln * 4;  // + 16h, h = 0..3

    // acc2[i][q]: row i, columns 2q and 2q+1 of the thread's 16 (q = 2h, 2h+1)
    uint64_t acc2[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc2[i][q] = 0ull;

    // slices counted in 32 bits (simt_supports keeps K below 2^33): with a
    // 64-bit counter this loop measured 1.5-5% slower (4096^3 and 4864 x
    // 4096 x 4096, both B layouts)
    const int n_slices = static_cast<int>((k_end - k_begin) / kWBK);
    fetch();
    stash(0);
    __syncthreads();
    for (int s = 0; s < n_slices; ++s) {
        const int buf = static_cast<int>(s & 1);
        const bool more = s + 1 < n_slices;
        float a[2][8];
        uint64_t b[2][8];
        auto frag = [&](int d, int k) {
            *reinterpret_cast<float4*>(&a[d][0]) = *reinterpret_cast<const float4*>(&sm.A[buf][k][am0]);
            *reinterpret_cast<float4*>(&a[d][4]) = *reinterpret_cast<const float4*>(&sm.A[buf][k][am1]);
#pragma unroll
            for (int h = 0; h < 4; ++h)
                *reinterpret_cast<ulonglong2*>(&b[d][2 * h]) =
                    *reinterpret_cast<const ulonglong2*>(&sm.B[buf][k][bn0 + h * 16]);
        };
        frag(0, 0);
#pragma unroll
        for (int k = 0; k < kWBK; ++k) {
            if (k == 2 && more) fetch();
            if (k + 1 < kWBK) frag((k + 1) & 1, k + 1);
            // the 8 broadcasts first, then the 64 packed FMAs column pair by
            // column pair: no FMA waits on the broadcast just made (measured
            // 64.9 -> 66.2 TFLOP/s at whole waves against rows outer)
            uint64_t ap[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ap[i] = pair_of(a[k & 1][i]);  // (a_i, a_i)
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
                for (int i = 0; i < 8; ++i) fma2(acc2[i][q], ap[i], b[k & 1][q]);
        }
        // the other buffer was last read in slice s-1, before the barrier that ended it
        if (more) stash(buf ^ 1);
        __syncthreads();
    }

    if (partial != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float* prow = partial + (i < 4 ? am0 + i : am1 + (i - 4)) * kWBN;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float v[4];
                unpair(acc2[i][2 * h], v[0], v[1]);
                unpair(acc2[i][2 * h + 1], v[2], v[3]);
                *reinterpret_cast<float4*>(prow + bn0 + h * 16) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + (i < 4 ? am0 + i : am1 + (i - 4));
        float* crow = p.C + r * p.ldc + col0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float v[4];
            unpair(acc2[i][2 * h], v[0], v[1]);
            unpair(acc2[i][2 * h + 1], v[2], v[3]);
            const int c = bn0 + h * 16;
            float4* dst = reinterpret_cast<float4*>(crow + c);
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kReadC) o = *dst;
            o.x = axpby(p.alpha, v[0], p.beta, o.x);
            o.y = axpby(p.alpha, v[1], p.beta, o.y);
            o.z = axpby(p.alpha, v[2], p.beta, o.z);
            o.w = axpby(p.alpha, v[3], p.beta, o.w);
            if (kBias) {
                const float4 bb = ld_f4(p.bias + col0 + c);
                o.x += bb.x;
                o.y += bb.y;
                o.z += bb.z;
                o.w += bb.w;
            }
            *dst = o;
        }
    }
}

// The wide schedule's whole tiles: block b owns tile b of the grouped order
// (every tile, or, under stream-K, the full_tiles tiles of the whole waves:
// blocks resident together work on neighbouring tiles, so they share A and B
// panels in L2).  The stream-K remainder is a kernel of its own
// (sgemm_wide_sk_kernel), so that each is compiled for its own loop alone;
// it is released as soon as every block here has started
// (griddepcontrol.launch_dependents) and its blocks take the SMs this grid's
// last wave frees.
template <bool kTransA, bool kTransB, int kReadC, int kBias>
__global__ void __launch_bounds__(kThreads, 1) sgemm_wide_kernel(Params p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) unsigned char wide_smem_raw[];
    WideSmem<kTransB>& sm = *reinterpret_cast<WideSmem<kTransB>*>(wide_smem_raw);
    int64_t tm, tn;
    wide_tile(blockIdx.x, p.M / kWBM, p.tiles_n, tm, tn);
    wide_block_tile<kTransA, kTransB, kReadC, kBias>(p, sm, tm * kWBM, tn * kWBN, 0, p.K, nullptr);
}

// The stream-K remainder (one block per SM, sk_ctas blocks): the tiles after
// the first full_tiles are shared out as units (tile t, K-slice s), in the
// order t * sk_slices + s, cut into sk_ctas equal contiguous ranges,
// u0(c) = c * sk_units / sk_ctas, so that every SM does the same work.  A
// tile a block covers whole gets the epilogue; a block's first and last
// segments, when they cover only part of a tile, go to the workspace as raw
// partial sums (slots 2c and 2c + 1, 128 x 256 floats each), and
// sgemm_wide_sk_reduce adds the pieces of each such tile in block order,
// i.e. in K order.  No block waits for another; each waits at its end for
// the whole-tile grid (griddepcontrol.wait), so that this grid completes
// after it and work behind it in the stream sees both.
template <bool kTransA, bool kTransB, int kReadC, int kBias>
__global__ void __launch_bounds__(kThreads, 1) sgemm_wide_sk_kernel(Params p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the reduce
    extern __shared__ __align__(16) unsigned char wide_smem_raw[];
    WideSmem<kTransB>& sm = *reinterpret_cast<WideSmem<kTransB>*>(wide_smem_raw);
    const int64_t tiles_m = p.M / kWBM;
    const int64_t c = blockIdx.x, S = p.sk_slices;
    const int64_t base = p.full_tiles * S;  // the first stream-K unit
    const int64_t u0 = base + c * p.sk_units / p.sk_ctas;
    const int64_t u1 = base + (c + 1) * p.sk_units / p.sk_ctas;
    for (int64_t u = u0; u < u1;) {
        const int64_t t = u / S, s0 = u - t * S;
        const int64_t end = min(u1, (t + 1) * S);
        const bool whole = s0 == 0 && end == (t + 1) * S;
        float* partial =
            whole ? nullptr : p.partials + (2 * c + (u == u0 ? 0 : 1)) * (kWBM * kWBN);
        int64_t tm, tn;
        wide_tile(t, tiles_m, p.tiles_n, tm, tn);
        wide_block_tile<kTransA, kTransB, kReadC, kBias>(p, sm, tm * kWBM, tn * kWBN,
                                                         s0 * kWBK, (end - t * S) * kWBK, partial);
        u = end;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The block whose stream-K range holds unit u (counted from the first
// stream-K unit): the largest c with c * units / ctas <= u.
__device__ __forceinline__ int64_t sk_owner(const Params& p, int64_t u) {
    return ((u + 1) * p.sk_ctas - 1) / p.sk_units;
}

// Adds the stream-K pieces of every tile split between blocks and applies
// the epilogue (float4 everywhere: the wide path runs only on aligned
// shapes).  Work item b = 1 .. sk_ctas - 1 is the range boundary between
// blocks b - 1 and b; the first boundary inside a tile handles that tile.
// kReduceSlabs blocks share a tile, 8 rows each, two float4 per thread.  The
// tile's pieces (the workspace slots of the blocks whose ranges meet it, in
// block order) are listed once per block; with at most kReducePieces of them
// every thread issues all its loads before adding them up, in block order
// (K order).  The block waits for the stream-K grid (griddepcontrol.wait)
// only after that set-up, so when it is launched as that grid's programmatic
// dependent its start overlaps the grid's end.
constexpr int kReduceSlabs = kWBM / 8;
constexpr int kReducePieces = 8;

__global__ void __launch_bounds__(kThreads) sgemm_wide_sk_reduce(Params p) {
    __shared__ int64_t s_slot[kReducePieces];
    __shared__ int s_pieces;  // < 0: the tile has more pieces than fit the list
    __shared__ int64_t s_first, s_last;
    const int64_t b = blockIdx.x / kReduceSlabs + 1;
    const int slab = static_cast<int>(blockIdx.x % kReduceSlabs);
    const int64_t S = p.sk_slices;
    // units counted from the first stream-K unit, tile T0 + T
    const int64_t ub = b * p.sk_units / p.sk_ctas;
    const int64_t T = ub / S;
    if (ub - T * S == 0) return;  // the boundary falls between tiles: nothing split here
    const int64_t prev = (b - 1) * p.sk_units / p.sk_ctas;
    if (b > 1 && prev / S == T && prev - T * S != 0) return;  // an earlier boundary owns T
    if (threadIdx.x == 0) {
        const int64_t c_first = sk_owner(p, T * S);
        const int64_t c_last = sk_owner(p, min((T + 1) * S, p.sk_units) - 1);
        int n = 0;
        for (int64_t q = c_first; q <= c_last; ++q) {
            // blocks with an empty range (fewer units than blocks) wrote nothing
            const int64_t q0 = q * p.sk_units / p.sk_ctas;
            if ((q + 1) * p.sk_units / p.sk_ctas == q0) continue;
            if (n == kReducePieces) {
                n = -1;
                break;
            }
            // block q's piece of T is its first segment if its range starts in T
            s_slot[n++] = 2 * q + (q0 / S == T ? 0 : 1);
        }
        s_pieces = n;
        s_first = c_first;
        s_last = c_last;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n = s_pieces;
    int64_t tm, tn;
    wide_tile(p.full_tiles + T, p.M / kWBM, p.tiles_n, tm, tn);
    const int64_t row0 = tm * kWBM, col0 = tn * kWBN;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = slab * (8 * kWBN / 4) + h * kThreads + threadIdx.x;
        const int r = e / (kWBN / 4), c = (e % (kWBN / 4)) * 4;
        const float* at = p.partials + r * kWBN + c;
        float4 sum;
        if (n > 0) {
            float4 v[kReducePieces];
#pragma unroll
            for (int i = 0; i < kReducePieces; ++i)
                if (i < n) v[i] = *reinterpret_cast<const float4*>(at + s_slot[i] * (kWBM * kWBN));
            sum = v[0];
#pragma unroll
            for (int i = 1; i < kReducePieces; ++i) {
                if (i < n) {
                    sum.x += v[i].x;
                    sum.y += v[i].y;
                    sum.z += v[i].z;
                    sum.w += v[i].w;
                }
            }
        } else {  // a long list: the same sum, one piece at a time
            sum = make_float4(0.f, 0.f, 0.f, 0.f);
            bool first = true;
            for (int64_t q = s_first; q <= s_last; ++q) {
                const int64_t q0 = q * p.sk_units / p.sk_ctas;
                if ((q + 1) * p.sk_units / p.sk_ctas == q0) continue;
                const int64_t slot = 2 * q + (q0 / S == T ? 0 : 1);
                const float4 w = *reinterpret_cast<const float4*>(at + slot * (kWBM * kWBN));
                if (first) {
                    sum = w;
                    first = false;
                } else {
                    sum.x += w.x;
                    sum.y += w.y;
                    sum.z += w.z;
                    sum.w += w.w;
                }
            }
        }
        float4* dst = reinterpret_cast<float4*>(p.C + (row0 + r) * p.ldc + col0 + c);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.beta != 0.0f) o = *dst;
        o.x = axpby(p.alpha, sum.x, p.beta, o.x);
        o.y = axpby(p.alpha, sum.y, p.beta, o.y);
        o.z = axpby(p.alpha, sum.z, p.beta, o.z);
        o.w = axpby(p.alpha, sum.w, p.beta, o.w);
        if (p.bias != nullptr) {
            const float4 bb = ld_f4(p.bias + col0 + c);
            o.x += bb.x;
            o.y += bb.y;
            o.z += bb.z;
            o.w += bb.w;
        }
        *dst = o;
    }
}

// The wide schedule for a problem of whole 128 x 256 tiles with at least one
// full wave of them (one block per SM); ok == false: not used.  A whole
// number of waves runs tile by tile; otherwise the whole waves and then the
// remainder stream-K, over one block per SM (sk_ctas), with 2 partial tiles
// per block of workspace (ws_bytes).
struct WidePlan {
    bool ok;
    int64_t tiles, tiles_n, slices;
    int64_t full_tiles;  // stream-K: the whole waves before the shared remainder
    int sk_ctas;  // 0: tile by tile
    size_t ws_bytes;
};

WidePlan plan_wide(const GemmArgs& a, int sm_count) {
    WidePlan w{};
    const bool shape = a.M % kWBM == 0 && a.N % kWBN == 0 && a.K % kWBK == 0 && a.K > 0 &&
                       a.lda % 4 == 0 && a.ldb % 4 == 0 && a.ldc % 4 == 0 &&
                       aligned(a.A, 16) && aligned(a.B, 16) && aligned(a.C, 16) &&
                       (a.bias == nullptr || aligned(a.bias, 16));
    if (!shape || sm_count <= 0) return w;
    w.tiles_n = a.N / kWBN;
    w.tiles = (a.M / kWBM) * w.tiles_n;
    w.slices = a.K / kWBK;
    if (w.tiles < sm_count || w.tiles > 0x7fffffff) return w;
    // units * ctas must not overflow 64 bits in the range arithmetic
    if (w.tiles > (INT64_MAX / sm_count) / w.slices) return w;
    w.ok = true;
    if (w.tiles % sm_count != 0) {
        w.sk_ctas = sm_count;
        w.full_tiles = w.tiles - w.tiles % sm_count;
        w.ws_bytes = static_cast<size_t>(2) * sm_count * kWBM * kWBN * sizeof(float);
    }
    return w;
}

// The whole-tile grid (blocks = its tiles), then, when sk is set, the
// stream-K grid (p.sk_ctas blocks) as its programmatic dependent.
template <bool kTransA, bool kTransB, int kReadC, int kBias>
cudaError_t launch_wide(const Params& p, int64_t blocks, bool sk, cudaStream_t s, int* launches) {
    const int smem = static_cast<int>(sizeof(WideSmem<kTransB>));
    auto kern = sgemm_wide_kernel<kTransA, kTransB, kReadC, kBias>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(blocks), kThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || !sk) return e;
    ++*launches;
    auto sk_kern = sgemm_wide_sk_kernel<kTransA, kTransB, kReadC, kBias>;
    e = cudaFuncSetAttribute(sk_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.sk_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sk_kern, p);
}

template <bool kTransA, bool kTransB>
cudaError_t launch_wide_layout(const Params& p, int64_t blocks, bool sk, bool read_c, bool bias,
                               cudaStream_t s, int* launches) {
    if (read_c && bias) return launch_wide<kTransA, kTransB, 1, 1>(p, blocks, sk, s, launches);
    if (read_c) return launch_wide<kTransA, kTransB, 1, 0>(p, blocks, sk, s, launches);
    if (bias) return launch_wide<kTransA, kTransB, 0, 1>(p, blocks, sk, s, launches);
    return launch_wide<kTransA, kTransB, 0, 0>(p, blocks, sk, s, launches);
}

}  // namespace

bool simt_supports(const GemmArgs& a) {
    // the kernels count K-slices (8 or 16 deep) in 32 bits
    return a.in_dtype == DGA_F32 && a.out_dtype == DGA_F32 && a.K < kSimtMaxK;
}

namespace {

template <bool kTransA, bool kTransB>
void launch_simt_kernels(const Params& p, const GemmArgs& a, const Schedule& sc, bool all_interior,
                         int64_t blocks) {
    if (all_interior) {
        dim3 grid(static_cast<unsigned>(a.N / BN), static_cast<unsigned>(a.M / BM));
        const bool rc = a.beta_f != 0.0f, bias = a.bias != nullptr;
        if (rc && bias)
            sgemm_128x128_interior_kernel<kSimtBlocksPerSm, kTransA, kTransB, 1, 1><<<grid, kThreads, 0, a.stream>>>(p);
        else if (rc)
            sgemm_128x128_interior_kernel<kSimtBlocksPerSm, kTransA, kTransB, 1, 0><<<grid, kThreads, 0, a.stream>>>(p);
        else if (bias)
            sgemm_128x128_interior_kernel<kSimtBlocksPerSm, kTransA, kTransB, 0, 1><<<grid, kThreads, 0, a.stream>>>(p);
        else
            sgemm_128x128_interior_kernel<kSimtBlocksPerSm, kTransA, kTransB, 0, 0><<<grid, kThreads, 0, a.stream>>>(p);
    } else {
        sgemm_128x128_kernel<kSimtBlocksPerSm, kTransA, kTransB>
            <<<static_cast<unsigned>(blocks), kThreads, 0, a.stream>>>(p);
    }
}

}  // namespace

namespace {

// Problems made only of interior tiles whose last wave is at most a third
// full run as two bands of whole tile rows: the top band (the full waves) on
// the interior kernel, the bottom band (the last wave) cut along K into 3-4
// parts by the general kernel over every slot.  Returns the top band's rows,
// or 0 for one band.  Measured on GB300 at N = K = 4096: whole waves run at
// 59 TFLOP/s; M = 3840 (last wave 16% full) went from 52.5 to 56.3 and
// M = 5120 (21%) from 54.8 to 57.7 with the bands, while M = 4096 (37%: its
// lone blocks already run ~1.8x faster than paired ones) lost 0.8% with a
// 2-way split and is left whole.
int64_t simt_top_band_rows(const GemmArgs& a, int sm_count, bool interior_shape) {
    if (!interior_shape) return 0;
    const int64_t tiles_n = a.N / BN, tiles = (a.M / BM) * tiles_n;
    const int64_t slots = static_cast<int64_t>(kSimtBlocksPerSm) * sm_count;
    if (slots <= 0 || tiles < slots) return 0;
    const int64_t tail = tiles % slots;
    if (tail == 0 || 3 * tail > slots) return 0;
    const int64_t rows = (tiles - tail) / tiles_n * BM;
    if (rows <= 0 || rows >= a.M) return 0;
    // the bottom band must itself be split at least 3 ways, else one band is as good
    if (plan_schedule(a.M - rows, a.N, a.K, sm_count).parts < 3) return 0;
    return rows;
}

bool simt_interior_shape(const GemmArgs& a) {
    return a.M % BM == 0 && a.N % BN == 0 && a.K % BK == 0 && a.lda % 4 == 0 && a.ldb % 4 == 0 &&
           a.ldc % 4 == 0 && aligned(a.A, 16) && aligned(a.B, 16) && aligned(a.C, 16);
}

cudaError_t simt_run(const GemmArgs& a, const DeviceInfo& dev, int* launches);

}  // namespace

size_t simt_workspace_size(const GemmArgs& a, int sm_count) {
    const WidePlan w = plan_wide(a, sm_count);
    if (w.ok) return w.ws_bytes;
    const int64_t top = simt_top_band_rows(a, sm_count, simt_interior_shape(a));
    return plan_schedule(a.M - top, a.N, a.K, sm_count).partial_bytes;
}

namespace {

// The wide kernel (and, for stream-K, its reduction) for a problem plan_wide
// accepted; stream_k false runs whole tiles, one block per tile.
cudaError_t wide_run(const GemmArgs& a, const WidePlan& w, bool stream_k, int* launches) {
    Params p{a.M, a.N, a.K, static_cast<const float*>(a.A), a.lda,
             static_cast<const float*>(a.B), a.ldb, static_cast<float*>(a.C), a.ldc,
             a.alpha_f, a.beta_f, 1, 1, 1, w.tiles_n, stream_k ? w.full_tiles : w.tiles, a.K, 1,
             stream_k ? static_cast<float*>(a.ws) : nullptr, static_cast<const float*>(a.bias),
             (w.tiles - w.full_tiles) * w.slices, w.slices, stream_k ? w.sk_ctas : 0};
    const int64_t blocks = stream_k ? w.full_tiles : w.tiles;
    const bool ta = a.layout_a == DGA_COL_MAJOR, tb = a.layout_b == DGA_COL_MAJOR;
    const bool rc = a.beta_f != 0.0f, bias = a.bias != nullptr;
    cudaError_t e;
    if (ta && tb) e = launch_wide_layout<true, true>(p, blocks, stream_k, rc, bias, a.stream, launches);
    else if (ta) e = launch_wide_layout<true, false>(p, blocks, stream_k, rc, bias, a.stream, launches);
    else if (tb) e = launch_wide_layout<false, true>(p, blocks, stream_k, rc, bias, a.stream, launches);
    else e = launch_wide_layout<false, false>(p, blocks, stream_k, rc, bias, a.stream, launches);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (stream_k) {
        // the reduce as a programmatic dependent of the stream-K grid
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>((w.sk_ctas - 1) * kReduceSlabs));
        cfg.blockDim = dim3(kThreads);
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, sgemm_wide_sk_reduce, p);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t simt_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches) {
    // Whole 128 x 256 tiles, at least one full wave: the wide kernel, with the
    // stream-K schedule when the waves are not whole and the workspace for it
    // was given.  Without that workspace a last wave at most half full goes
    // to the 128 x 128 kernel below (one block per SM would idle most SMs for
    // a whole tile time), a fuller one stays on the wide kernel, whole tiles.
    const WidePlan w = plan_wide(a, dev.sm_count);
    if (w.ok) {
        if (w.sk_ctas == 0) return wide_run(a, w, false, launches);
        if (a.ws != nullptr && a.ws_bytes >= w.ws_bytes) return wide_run(a, w, true, launches);
        if (2 * (w.tiles % dev.sm_count) > dev.sm_count) return wide_run(a, w, false, launches);
    }
    const int64_t top = simt_top_band_rows(a, dev.sm_count, simt_interior_shape(a));
    if (top > 0 && a.ws != nullptr &&
        a.ws_bytes >= plan_schedule(a.M - top, a.N, a.K, dev.sm_count).partial_bytes) {
        GemmArgs upper = a, lower = a;
        upper.M = top;
        lower.M = a.M - top;
        lower.A = a.layout_a == DGA_COL_MAJOR ? static_cast<const float*>(a.A) + top
                                              : static_cast<const float*>(a.A) + top * a.lda;
        lower.C = static_cast<float*>(a.C) + top * a.ldc;
        cudaError_t e = simt_run(upper, dev, launches);
        if (e != cudaSuccess) return e;
        return simt_run(lower, dev, launches);
    }
    return simt_run(a, dev, launches);
}

namespace {

cudaError_t simt_run(const GemmArgs& a, const DeviceInfo& dev, int* launches) {
    Schedule sc = plan_schedule(a.M, a.N, a.K, dev.sm_count);
    if (sc.parts > 1 && (a.ws == nullptr || a.ws_bytes < sc.partial_bytes)) {
        // not enough workspace for the split tail: whole tiles only
        sc.full_tiles = sc.tiles;
        sc.parts = 1;
        sc.part_k = a.K;
    }
    Params p{a.M, a.N, a.K, static_cast<const float*>(a.A), a.lda,
             static_cast<const float*>(a.B), a.ldb, static_cast<float*>(a.C), a.ldc,
             a.alpha_f, a.beta_f, (a.ldc % 4 == 0 && aligned(a.C, 16)) ? 1 : 0,
             (a.lda % 4 == 0 && aligned(a.A, 16)) ? 1 : 0, (a.ldb % 4 == 0 && aligned(a.B, 16)) ? 1 : 0,
             sc.tiles_n, sc.full_tiles, sc.part_k, sc.parts,
             sc.parts > 1 ? static_cast<float*>(a.ws) : nullptr, static_cast<const float*>(a.bias)};
    const int64_t tail = sc.tiles - sc.full_tiles;
    const int64_t blocks = sc.full_tiles + tail * sc.parts;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const bool all_interior = sc.parts == 1 && a.M % BM == 0 && a.N % BN == 0 && a.K % BK == 0 &&
                              p.vec_a && p.vec_b && p.vec_c && a.M / BM <= 65535 &&
                              a.N / BN <= 0x7fffffff;
    const bool ta = a.layout_a == DGA_COL_MAJOR, tb = a.layout_b == DGA_COL_MAJOR;
    if (ta && tb) launch_simt_kernels<true, true>(p, a, sc, all_interior, blocks);
    else if (ta) launch_simt_kernels<true, false>(p, a, sc, all_interior, blocks);
    else if (tb) launch_simt_kernels<false, true>(p, a, sc, all_interior, blocks);
    else launch_simt_kernels<false, false>(p, a, sc, all_interior, blocks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
    if (tail > 0 && sc.parts > 1) {
        sgemm_tail_reduce<<<static_cast<unsigned>(tail * kTailSlabs), kThreads, 0, a.stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace

}  // namespace dga
