// gemv_skinny.cu -- the bandwidth-bound path for skinny products
//     Y[M, N] = alpha * X[M, K] * W[N, K]^T + beta * Y (+ bias),   M <= 16,
// i.e. dga_gemm with A = X (row-major), B column-major (W stored N x K, the
// Linear-layer weight layout of "AI Programming: Matrix Product", section
// "Fully-connected layer") and C = Y.
//
// Why a separate path: a GEMV moves 2 bytes of weight per multiply-add, so no
// amount of arithmetic speed helps; the time is the weight's bytes divided
// by HBM bandwidth ("Matrix multiplication: arithmetic intensity, tiling and
// Tensor Core", section 5.1, the matrix-vector row of its table, and section
// 5.6).  The design therefore only has to (1) read every weight byte exactly
// once with enough bytes in flight, and (2) keep the arithmetic off the
// critical path.
//
//  * Rows: the grid is a whole number of waves of one CTA per SM, and the N
//    weight rows are shared out evenly (8192 rows on 152 SMs: 53 or 54 rows
//    per CTA, at most 64), so every SM streams the same number of bytes.
//  * Streaming: a producer warp issues TMA loads into a ring of stages in
//    shared memory; a stage holds 256 k of the CTA's weight rows (four boxes
//    of 64 k x rows, 128-byte swizzle) and of the M <= 16 activation rows
//    (four boxes of 64 k x 16 rows; rows past M are zero-filled by TMA).
//    Boxes of a CTA's own rows and a ring of about 180 KB keep ~150 KB of
//    weights in flight per SM: on GB300 this streams a 128 MB matrix at
//    ~87% of the measured copy bandwidth, where per-lane 16-byte cp.async
//    copies of the same rows reach ~80%.
//  * Arithmetic: 8 consumer warps, one per (16-row tile, half of the stage's
//    16 k-steps), multiply with mma.sync m16n8k16 (weight rows = MMA M,
//    activation rows = MMA N, fp32 accumulate), fragments read by ldmatrix
//    from the swizzled boxes (the swizzle makes those reads conflict-free).
//    A warp releases a stage by arriving on its "empty" mbarrier; the
//    producer refills the slot once all 8 have, so no warp waits for another
//    between stages.  (tcgen05 was tried here: an M = 128, N = 16 MMA per
//    16 k costs about 117 cycles, which made the stream 30% slower.)
//  * Each CTA starts its walk over K at a different stage, so the CTAs do not
//    all read the same activation lines at the same moment.
//  * At the end each output has two partial sums, held by the two warps of
//    its tile: one warp hands its fragments over through 4 KB of shared
//    memory and the other applies alpha, beta and the bias and stores from
//    the MMA fragment layout.  (Splitting k-steps over all 8 warps instead
//    made the 8-way reduction of 64 rows x 16 outputs cost ~1.5 us of a
//    25 us kernel at M = 16.)
//  * Launched with programmatic stream serialization: the next kernel on the
//    stream may be launched while this one drains, but every thread waits
//    (griddepcontrol.wait) for the previous grid to complete and its writes
//    to become visible before touching global memory, so results and stream
//    order are exactly those of a plain launch; back-to-back calls only
//    overlap launch and set-up with the previous call's tail.
//  * Every wait is bounded; a wait that expires records a code in this
//    family's status word (read by dga_sync_status) and the CTA returns after
//    its copies in flight have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "dga_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace dga {

__device__ int g_skinny_status;  // non-zero: a bounded wait expired (role code)

namespace {

constexpr int kBoxK = 64;                 // k per TMA box: one 128-byte swizzle row
constexpr int kBoxesPerStage = 4;         // 256 k per stage
constexpr int kXRows = 16;                // activation rows per box (M <= 16)
constexpr int kMaxRows = 64;              // weight rows per CTA: 4 MMA m-tiles
constexpr uint32_t kXBoxBytes = kXRows * kBoxK * 2;      // 2 KB
constexpr uint32_t kRingBudget = 216 * 1024;             // bytes of stages (6 of 36 KB at 54 rows)
constexpr int kMaxStages = 8;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;      // + one producer warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;         // 2 s
constexpr uint32_t kBarrierBytes = 2 * kMaxStages * 8 + 16;  // full[], empty[], abort flag
constexpr uint32_t kRedBytes = (kMaxRows / 16) * 2 * 32 * 16;  // 4 tiles x MT <= 2 x 32 lanes x float4

enum : int { kRoleProducer = 1, kRoleConsumer = 2 };

struct Params {
    int64_t M, N, K;
    void* Y;
    int64_t ldy;
    float alpha, beta;
    const void* bias;      // N output-type values added to every row, or null
    int64_t ctas;          // grid size: CTA c owns rows [c*N/ctas, (c+1)*N/ctas)
    uint32_t rows_lo;      // floor(N / ctas): rows of the short CTAs (box of map lo)
    uint32_t w_box_bytes;  // stride of the weight boxes: (rows_lo + 1) * 128 rounded to 1 KB
    uint32_t stages;       // ring stages (<= kMaxStages)
    uint32_t n_kstages;    // ceil(K / 256)
};

__host__ __device__ inline uint32_t stage_bytes(uint32_t w_box_bytes) {
    return kBoxesPerStage * (w_box_bytes + kXBoxBytes);
}

__device__ __forceinline__ void record_failure(int role, volatile int* abort_flag) {
    atomicCAS(&g_skinny_status, 0, role);
    *abort_flag = 1;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(saddr));
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

// Shared-memory address of the 16-byte chunk `chunk` (0..7) of row `row` of a
// box written by TMA with the 128-byte swizzle (rows of 128 bytes, box base
// 1024-byte aligned): the chunk index is XORed with the row's index in its
// group of 8 rows.
__device__ __forceinline__ uint32_t sw128(uint32_t box, uint32_t row, uint32_t chunk) {
    return box + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Shared memory (dynamic, 1024-byte aligned): stages of
//   [W box 0][W box 1][W box 2][W box 3][X box 0][X box 1][X box 2][X box 3]
// then the barriers, then the 4 KB hand-over area of the final reduction.
// MT = 8-row activation tiles (1 for M <= 8, 2 for M <= 16).
template <bool kBf16, int MT, typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap tmW_lo, const __grid_constant__ CUtensorMap tmW_hi,
                  const __grid_constant__ CUtensorMap tmX, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbytes = stage_bytes(p.w_box_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * sbytes);
    uint64_t* empty = full + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxStages);
    // partial sums handed from the second warp of a tile to the first
    float4* red = reinterpret_cast<float4*>(smem + p.stages * sbytes + kBarrierBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * p.N / p.ctas;
    const int64_t n_end = (static_cast<int64_t>(blockIdx.x) + 1) * p.N / p.ctas;
    const uint32_t rows = static_cast<uint32_t>(n_end - n0);  // rows_lo or rows_lo + 1
    const int rt_used = static_cast<int>((rows + 15) / 16);   // m-tiles holding rows

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the previous grid on the stream has completed and its writes are visible
    // past this point; let the next one be scheduled
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // CTAs start at different K stages (fixed per CTA: results stay deterministic)
    const uint32_t k_start = static_cast<uint32_t>(blockIdx.x % p.n_kstages);

    float acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.0f;
    const int tile = warp & 3, khalf = warp >> 2;  // consumer warps: 16-row tile, k-step half

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const CUtensorMap* tmW = rows == p.rows_lo ? &tmW_lo : &tmW_hi;
            const uint32_t tx_bytes = kBoxesPerStage * (rows * kBoxK * 2 + kXBoxBytes);
            tma_prefetch_desc(tmW);
            tma_prefetch_desc(&tmX);
            uint32_t stage = 0, phase = 0;
            uint32_t issued_phase[kMaxStages];
            bool issued[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued[s] = false;
            for (uint32_t i = 0; i < p.n_kstages; ++i) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, kWaitLimitNs)) {
                    record_failure(kRoleProducer, abort_flag);
                    break;
                }
                uint32_t ks = i + k_start;
                if (ks >= p.n_kstages) ks -= p.n_kstages;
                uint8_t* base = smem + stage * sbytes;
                mbar_arrive_expect_tx(&full[stage], tx_bytes);
                for (int b = 0; b < kBoxesPerStage; ++b) {
                    const int32_t k0 = static_cast<int32_t>((ks * kBoxesPerStage + b) * kBoxK);
                    tma_load_2d(base + b * p.w_box_bytes, tmW, &full[stage], k0,
                                static_cast<int32_t>(n0));
                    tma_load_2d(base + kBoxesPerStage * p.w_box_bytes + b * kXBoxBytes, &tmX,
                                &full[stage], k0, 0);
                }
                issued[stage] = true;
                issued_phase[stage] = phase;
                if (++stage == p.stages) { stage = 0; phase ^= 1; }
            }
            // copies still in flight must land before the ring is reused
            for (uint32_t s = 0; s < p.stages; ++s)
                if (issued[s]) {
                    volatile int never = 0;
                    mbar_wait_bounded(&full[s], issued_phase[s], &never, kWaitLimitNs);
                }
        }
    } else {
        // ------------------------------------------------ consumer warps
        // warp w: rows [16 * (w % 4), +16) and k-steps [8 * (w / 4), +8) of
        // every stage (k-step s: box s / 4, 16-byte chunks 2 (s % 4), +1)
        const bool active = tile < rt_used;
        const uint32_t a_row = lane & 15, a_half = lane >> 4;
        const uint32_t b_row = lane & 7, b_half = (lane >> 3) & 1;
        uint32_t stage = 0, phase = 0;
        for (uint32_t i = 0; i < p.n_kstages; ++i) {
            if (!mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitLimitNs)) {
                if (lane == 0) record_failure(kRoleConsumer, abort_flag);
                break;
            }
            const uint32_t base = smem_u32(smem + stage * sbytes);
            if (active) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t ks = khalf * 8 + j, box = ks >> 2, c0 = (ks & 3) * 2;
                    const uint32_t wbox = base + box * p.w_box_bytes;
                    const uint32_t xbox = base + kBoxesPerStage * p.w_box_bytes + box * kXBoxBytes;
                    uint32_t a[4];
                    ldmatrix_x4(a, sw128(wbox, tile * 16 + a_row, c0 + a_half));
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        uint32_t b[2];
                        ldmatrix_x2(b, sw128(xbox, m * 8 + b_row, c0 + b_half));
                        mma16816<kBf16>(acc[m], a, b[0], b[1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == p.stages) { stage = 0; phase ^= 1; }
        }
    }
    if (warp == kConsumerWarps) return;  // the producer has waited for its copies
    const bool active = tile < rt_used;
    if (active && khalf == 1) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            red[(tile * MT + m) * 32 + lane] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");  // consumer warps only
    if (!active || khalf == 1 || *abort_flag) return;

    // D fragment of n-tile m: acc[m][2h + j] is weight row g + 8h of the
    // tile (output column n) and activation row 8m + 2t + j (output row)
    const int g = lane >> 2, t = lane & 3;
    TOut* Y = static_cast<TOut*>(p.Y);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float4 o = red[(tile * MT + m) * 32 + lane];
        const float v[4] = {acc[m][0] + o.x, acc[m][1] + o.y, acc[m][2] + o.z, acc[m][3] + o.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t row = tile * 16 + g + 8 * h;
            if (row >= rows) continue;
            const int64_t n = n0 + row;
            const float bv = p.bias ? OutT<TOut>::load(static_cast<const TOut*>(p.bias) + n) : 0.0f;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int act = m * 8 + 2 * t + j;
                if (act >= p.M) continue;
                TOut* dst = Y + act * p.ldy + n;
                const float old = p.beta != 0.0f ? OutT<TOut>::load(dst) : 0.0f;
                OutT<TOut>::store(dst, axpby(p.alpha, v[2 * h + j], p.beta, old) + bv);
            }
        }
    }
}

// ---- host side -------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// rows x K 16-bit elements, row stride ld; boxes of 64 k x box_rows, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ld,
                     uint32_t box_rows, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// CTAs: whole waves of one CTA per SM, as few as keep every CTA at <= 64
// rows, but no more CTAs than 16-row groups.
int64_t skinny_ctas(int64_t N, int sm_count) {
    const int64_t sms = sm_count > 0 ? sm_count : 1;
    const int64_t min_ctas = (N + kMaxRows - 1) / kMaxRows;
    const int64_t waves = (min_ctas + sms - 1) / sms;
    return std::max<int64_t>(1, std::min(waves * sms, (N + 15) / 16));
}

template <bool kBf16, int MT, typename TOut>
cudaError_t launch_mt(const CUtensorMap& lo, const CUtensorMap& hi, const CUtensorMap& x,
                      const Params& p, int smem, cudaStream_t s) {
    auto kern = skinny_kernel<kBf16, MT, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, lo, hi, x, p);
}

template <bool kBf16, typename TOut>
cudaError_t launch_typed(const CUtensorMap& lo, const CUtensorMap& hi, const CUtensorMap& x,
                         const Params& p, int smem, cudaStream_t s) {
    return p.M <= 8 ? launch_mt<kBf16, 1, TOut>(lo, hi, x, p, smem, s)
                    : launch_mt<kBf16, 2, TOut>(lo, hi, x, p, smem, s);
}

}  // namespace

bool skinny_supports(const GemmArgs& a) {
    const bool types = (a.in_dtype == DGA_BF16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_BF16)) ||
                       (a.in_dtype == DGA_F16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_F16));
    // TMA: 16-byte row strides and bases, 32-bit extents
    return types && a.layout_a == DGA_ROW_MAJOR && a.layout_b == DGA_COL_MAJOR && a.M >= 1 &&
           a.M <= kXRows && a.K >= 1 && a.K < (int64_t(1) << 31) && a.N < (int64_t(1) << 31) &&
           a.lda % 8 == 0 && a.ldb % 8 == 0 && aligned(a.A, 16) && aligned(a.B, 16) &&
           encode_fn() != nullptr;
}

cudaError_t skinny_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches) {
    Params p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.Y = a.C;
    p.ldy = a.ldc;
    p.alpha = a.alpha_f;
    p.beta = a.beta_f;
    p.bias = a.bias;
    p.ctas = skinny_ctas(a.N, dev.sm_count);
    if (p.ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    p.rows_lo = static_cast<uint32_t>(a.N / p.ctas);                   // >= 1, <= 64
    const uint32_t rows_hi = std::min<uint32_t>(p.rows_lo + 1, kMaxRows);
    p.w_box_bytes = (rows_hi * kBoxK * 2 + 1023) / 1024 * 1024;
    p.stages = std::min<uint32_t>(kMaxStages, kRingBudget / stage_bytes(p.w_box_bytes));
    p.n_kstages = static_cast<uint32_t>((a.K + kBoxK * kBoxesPerStage - 1) / (kBoxK * kBoxesPerStage));
    // ring + barriers + the hand-over area of the final reduction + alignment slack
    const int smem = static_cast<int>(p.stages * stage_bytes(p.w_box_bytes) + kBarrierBytes +
                                      kRedBytes + 1024);
    if (p.stages < 2 || smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;

    const bool bf = a.in_dtype == DGA_BF16;
    CUtensorMap lo, hi, x;
    cudaError_t e = make_map(&lo, a.B, a.N, a.K, a.ldb, p.rows_lo, bf);
    if (e == cudaSuccess) e = make_map(&hi, a.B, a.N, a.K, a.ldb, rows_hi, bf);
    if (e == cudaSuccess) e = make_map(&x, a.A, a.M, a.K, a.lda, kXRows, bf);
    if (e != cudaSuccess) return e;

    if (a.out_dtype == DGA_F32) e = bf ? launch_typed<true, float>(lo, hi, x, p, smem, a.stream)
                                       : launch_typed<false, float>(lo, hi, x, p, smem, a.stream);
    else if (a.out_dtype == DGA_BF16) e = launch_typed<true, __nv_bfloat16>(lo, hi, x, p, smem, a.stream);
    else if (a.out_dtype == DGA_F16) e = launch_typed<false, __half>(lo, hi, x, p, smem, a.stream);
    else e = cudaErrorInvalidValue;
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t skinny_status_take(int* status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_skinny_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v != 0) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_skinny_status, &zero, sizeof zero);
    }
    *status = v;
    return e;
}

}  // namespace dga
