// gemm_tcgen05.cu -- GEMM on the 5th-generation tensor cores of sm_103a.
//
// What it computes: C <- alpha * A * B + beta * C with bf16 or fp16 inputs,
// fp32 accumulation and fp32 / bf16 / fp16 output -- the Tensor Core
// precision rows (BF16 / FP16 inputs, FP32 accumulate) of "Matrix
// multiplication: arithmetic intensity, tiling and Tensor Core", section
// 5.5 -- and, on request only, fp32 inputs multiplied as TF32 (the TF32 row
// of the same table; 10 mantissa bits, so lossy, as section 5.7 warns).  The pages' own tensor-core kernels are WMMA 16x16x16 warp tiles on
// A100/H100; this one is built for Blackwell instead:
//
//   * One persistent CTA per SM walks output tiles of 128 x 256 in a grouped
//     order (a group of tile rows sized so its A panels stay in L2) so that
//     concurrently running tiles share A and B panels in L2.
//   * Warp 0 (one lane) is the TMA producer: 2-D tensor-map loads of a
//     128 x 64 A box and a 256 x 64 B box (64 bf16 = one 128-byte swizzle
//     row) into a 4-stage shared-memory ring, each stage guarded by a
//     "full" and an "empty" mbarrier.  Out-of-range rows and the K tail are
//     filled with zeros by the TMA unit, which is the zero-fill edge rule of
//     "AI Programming: Matrix Product", section "Shared Memory Tiling".
//   * Warp 1 (one lane) issues tcgen05.mma (M = 128, N = 256, K = 16; four per
//     stage) into an fp32 accumulator in tensor memory, and tcgen05.commit to
//     release each stage and, after the last K block, the accumulator.
//   * Warps 2-5 are the epilogue (INT8: warps 2-17, see below): tcgen05.ld moves the accumulator to
//     registers, 32 columns at a time, for the fused alpha/beta update and the
//     masked store.  TMEM holds two accumulators (2 x 256 of its 512
//     columns), so the epilogue of tile i overlaps the main loop of tile i+1.
//   * Every wait is bounded in time; a wait that expires records a code in a
//     per-device status word, tells the other roles to stop, and the CTA
//     drains its outstanding copies and MMAs and frees its TMEM before
//     returning (read with dga_sync_status()).
//
// TF32 uses the same kernels with kind::tf32: a K block is still one
// 128-byte swizzle row (32 fp32 elements instead of 64 16-bit ones) and every
// MMA still consumes 32 bytes of it (K = 8 instead of 16), so the shared
// memory layout, descriptors and pipeline are the same.  TF32 operands are
// always read K-major: a column-major A or row-major B is first transposed
// into the workspace by pack_transposed_f32_kernel.
//
// Operands reach the tensor cores in their own layout: K-major (A row-major,
// B column-major) as 64 x rows boxes, or MN-major (A column-major, B
// row-major: the G^T and W of a fully-connected layer's gradients) as boxes of
// 64 MN-elements x 64 k, one per 64 rows of the tile, read by the MMA through
// MN-major descriptors (transpose bits of the instruction descriptor).  Only
// a leading dimension TMA cannot express (not a multiple of 16 bytes, or an
// unaligned base) and INT8 inputs (encoded exactly as bf16, see below) are
// first repacked into the caller's workspace, both operands by one launch of
// pack_pair_kernel that the GEMM follows as a programmatic dependent.
//
// INT8 x INT8 -> INT32 (tcgen05 has no integer MMA on sm_103a: ptxas rejects
// kind::i8 for this target).  Every int8 value is an exact bf16, every
// product of two is an integer of magnitude <= 2^14, and the tensor core
// accumulates in fp32.  The K loop is cut into chunks of 1024: within a chunk
// every partial sum is an integer of magnitude <= 1024 * 2^14 = 2^24, and
// fp32 represents every integer of that magnitude exactly, so each chunk's
// fp32 accumulator holds the exact integer chunk sum.  The epilogue converts
// each chunk result to int32 (exact) and adds it into int32 registers
// (two's-complement wrap), so the final sum is exact for any K.  Sixteen
// epilogue warps (64 columns each) drain a chunk while the MMA fills the
// other accumulator; longer chunks mean fewer of these hand-offs (1024
// measured 15% faster than 256 at 4093 x 4099 x 4096).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "dga_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace dga {

__device__ int g_tc_status;  // non-zero: a bounded wait expired (role code)

namespace {

constexpr int BM = 128;  // tile rows (UMMA M)
constexpr int BK = 64;   // 16-bit K elements per stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int UK = 16;   // 16-bit K elements per tcgen05.mma (32 bytes; kind::f16)
// K elements per stage for an operand format: 32 fp32 elements for TF32.
__host__ __device__ constexpr int k_per_stage(uint32_t fmt) { return fmt == kFmtTF32 ? BK / 2 : BK; }
constexpr int kStages = 4;
constexpr int kI8ChunkBlocks = 16;  // INT8: K blocks per exact fp32 chunk (16 x 64 = 1024)
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s
constexpr uint32_t kMnAtom = 64;                        // MN-elements per MN-major box
constexpr uint32_t kMnBoxBytes = kMnAtom * BK * 2;      // one 64 x 64 box: 8 KB
// Descriptor start-address steps (16-byte units) per K = 16 MMA: 32 bytes
// along the swizzle row when K-major, 16 k-rows of 128 bytes when MN-major.
constexpr uint32_t kStepKMajor = (UK * 2) >> 4;
constexpr uint32_t kStepMnMajor = (UK * 128) >> 4;
static_assert(BM % kMnAtom == 0, "MN-major A boxes tile the block rows");

enum : int { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleSelfTest = 4 };

struct TcParams {
    int64_t M, N, K;
    void* C;
    int64_t ldc;
    float alpha, beta;
    int32_t alpha_i, beta_i;
    const void* bias;  // N output-type (int32 for INT8) values added to every row, or null
    uint32_t a_mn, b_mn;  // operand stored MN-major (column-major A / row-major B)
    uint32_t tiles_m, tiles_n, num_tiles, num_kb;
    uint32_t group_m;  // tile rows per raster group
    // CTA-pair kernel, floating point: the tiles after the first full_tiles
    // (the last, part-filled wave) are each cut along K into `splits` parts,
    // one work unit each, whose raw fp32 sums go to `partials` (256 x 256
    // words per unit) for tc_split_reduce_kernel;
    // num_units = full_tiles + (num_tiles - full_tiles) * splits.
    // splits == 1: every unit is a tile.
    uint32_t full_tiles, splits, num_units;
    uint32_t* partials;
};

// Shared-memory plan (dynamic, 1024-byte aligned): the stage ring, the
// barriers, then one 32 x 33 staging square per epilogue warp (the padding
// column keeps both the row-wise writes and the column-wise reads free of
// bank conflicts).  BN is the tile width; kSquares is 4 for floating point
// (one per epilogue warp) and 8 for INT8, whose 16 epilogue warps share them
// in two rounds.
template <int BN, int kSquares>
struct Smem {
    static constexpr uint32_t kABytes = BM * BK * 2;
    static constexpr uint32_t kBBytes = BN * BK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kRing = kStages * kStageBytes;
    static constexpr uint32_t kBarOffset = kRing;
    // full[S], empty[S], acc_full[2], acc_empty[2], drain, then tmem slot + abort flag
    static constexpr uint32_t kBarBytes = (2 * kStages + 5) * 8 + 16;
    static constexpr uint32_t kEpiOffset = (kBarOffset + kBarBytes + 127) / 128 * 128;
    static constexpr uint32_t kEpiWarpBytes = 32 * 33 * 4;
    static constexpr uint32_t kTotal = kEpiOffset + kSquares * kEpiWarpBytes;
    static constexpr uint32_t kLaunchBytes = kTotal + 1024;  // + alignment slack
};

__device__ __forceinline__ void tile_coords(uint32_t t, const TcParams& p, uint32_t& tm,
                                            uint32_t& tn) {
    const uint32_t group_size = p.group_m * p.tiles_n;
    const uint32_t group = t / group_size;
    const uint32_t first_m = group * p.group_m;
    const uint32_t gm = min(p.tiles_m - first_m, p.group_m);
    const uint32_t r = t % group_size;
    tm = first_m + r % gm;
    tn = r / gm;
}

// Work unit u of the CTA-pair kernel: its tile, its k-blocks [kb_begin,
// kb_end) and, for a part of a split tile, its partial-sum slot (else -1).
__device__ __forceinline__ void unit_coords(uint32_t u, const TcParams& p, uint32_t& tm,
                                            uint32_t& tn, uint32_t& kb_begin, uint32_t& kb_end,
                                            int32_t& slot) {
    uint32_t t = u;
    kb_begin = 0;
    kb_end = p.num_kb;
    slot = -1;
    if (u >= p.full_tiles) {
        const uint32_t v = u - p.full_tiles, part = v % p.splits;
        t = p.full_tiles + v / p.splits;
        kb_begin = part * p.num_kb / p.splits;
        kb_end = (part + 1) * p.num_kb / p.splits;
        slot = p.splits > 1 ? static_cast<int32_t>(v) : -1;
    }
    tile_coords(t, p, tm, tn);
}

__device__ __forceinline__ void record_failure(int role, volatile int* abort_flag) {
    atomicCAS(&g_tc_status, 0, role);
    *abort_flag = 1;
}

// ---- epilogue stores ---------------------------------------------------------
//
// A warp holds a 32 x 32 block of the tile: lane l has row (row_base + l),
// columns col_base + j in v[j].  Storing that directly would make every store
// instruction touch 32 different rows.  The block is therefore transposed
// through shared memory, so that each store instruction writes 32
// consecutive elements of one row (whole 32-byte sectors), whatever the
// alignment of C or ldc.

template <typename TOut>
__device__ __forceinline__ void store_block_staged(const TcParams& p, uint32_t* stage, int lane,
                                                   int64_t row_base, int64_t col_base,
                                                   const uint32_t (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = v[j];
    __syncwarp();
    const int64_t col = col_base + lane;
    const bool col_ok = col < p.N;
    const float bv = (p.bias != nullptr && col_ok) ? OutT<TOut>::load(static_cast<const TOut*>(p.bias) + col) : 0.0f;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
        const int64_t row = row_base + i;
        if (col_ok && row < p.M) {
            TOut* dst = static_cast<TOut*>(p.C) + row * p.ldc + col;
            const float old = p.beta != 0.0f ? OutT<TOut>::load(dst) : 0.0f;
            OutT<TOut>::store(dst, axpby(p.alpha, __uint_as_float(stage[i * 33 + lane]), p.beta, old) + bv);
        }
    }
    __syncwarp();  // the next block reuses the square
}

__device__ __forceinline__ void store_block_staged_i32(const TcParams& p, uint32_t* stage,
                                                       int lane, int64_t row_base,
                                                       int64_t col_base, const int32_t* v) {
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = static_cast<uint32_t>(v[j]);
    __syncwarp();
    const int64_t col = col_base + lane;
    const bool col_ok = col < p.N;
    const uint32_t bv = (p.bias != nullptr && col_ok) ? static_cast<uint32_t>(static_cast<const int32_t*>(p.bias)[col]) : 0u;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
        const int64_t row = row_base + i;
        if (col_ok && row < p.M) {
            int32_t* dst = static_cast<int32_t*>(p.C) + row * p.ldc + col;
            const int32_t old = p.beta_i != 0 ? *dst : 0;
            const int32_t v = axpby_i32(p.alpha_i, static_cast<int32_t>(stage[i * 33 + lane]), p.beta_i, old);
            *dst = static_cast<int32_t>(static_cast<uint32_t>(v) + bv);
        }
    }
    __syncwarp();
}

// ---- the kernel ----------------------------------------------------------------
//
// kI8: INT8 mode (bf16-encoded operands, chunked exact accumulation, int32 out).
// BN: tile columns.  Epilogue warps: 4 (float) or 8 (INT8: two column halves).

template <uint32_t kFmt, bool kI8, int BN, typename TOut>
__global__ void __launch_bounds__(kI8 ? 576 : 192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   TcParams p) {
    constexpr int kEpiWarps = kI8 ? 16 : 4;
    static_assert(BN % kMnAtom == 0, "MN-major B boxes tile the block columns");
    using S = Smem<BN, kI8 ? 8 : 4>;
    constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
    constexpr uint32_t kIdesc = idesc_mma(kFmt, BM, BN);
    constexpr int kKElems = k_per_stage(kFmt);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps * 32);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // launched right behind the operand repack (programmatic serialisation):
    // everything above overlapped its tail; its output is read only from here
    // on (a no-op when the launch has no such dependency)
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; ++s) issued[s] = false;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
                uint32_t tm, tn;
                tile_coords(t, p, tm, tn);
                for (uint32_t kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, kWaitLimitNs)) {
                        record_failure(kRoleProducer, abort_flag);
                        ok = false;
                        break;
                    }
                    uint8_t* a_dst = smem + stage * S::kStageBytes;
                    uint8_t* b_dst = a_dst + S::kABytes;
                    mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
                    const int32_t k0 = static_cast<int32_t>(kb * kKElems);
                    if (p.a_mn) {
                        for (uint32_t j = 0; j < BM / kMnAtom; ++j)
                            tma_load_2d(a_dst + j * kMnBoxBytes, &tmA, &full[stage],
                                        static_cast<int32_t>(tm * BM + j * kMnAtom), k0);
                    } else {
                        tma_load_2d(a_dst, &tmA, &full[stage], k0, static_cast<int32_t>(tm * BM));
                    }
                    if (p.b_mn) {
                        for (uint32_t j = 0; j < BN / kMnAtom; ++j)
                            tma_load_2d(b_dst + j * kMnBoxBytes, &tmB, &full[stage],
                                        static_cast<int32_t>(tn * BN + j * kMnAtom), k0);
                    } else {
                        tma_load_2d(b_dst, &tmB, &full[stage], k0, static_cast<int32_t>(tn * BN));
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            // Copies still in flight must land before shared memory goes away.
            for (int s = 0; s < kStages; ++s)
                if (issued[s]) {
                    volatile int never = 0;
                    mbar_wait_bounded(&full[s], issued_phase[s], &never, kWaitLimitNs);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            const uint32_t idesc = idesc_major(kIdesc, p.a_mn, p.b_mn);
            const uint32_t a_step = p.a_mn ? kStepMnMajor : kStepKMajor;
            const uint32_t b_step = p.b_mn ? kStepMnMajor : kStepKMajor;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
                const uint32_t n_chunks = kI8 ? (p.num_kb + kI8ChunkBlocks - 1) / kI8ChunkBlocks : 1;
                for (uint32_t ch = 0; ok && ch < n_chunks; ++ch) {
                    if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1, abort_flag, kWaitLimitNs)) {
                        record_failure(kRoleMma, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * BN;
                    const uint32_t kb_begin = kI8 ? ch * kI8ChunkBlocks : 0;
                    const uint32_t kb_end = kI8 ? min(p.num_kb, kb_begin + kI8ChunkBlocks) : p.num_kb;
                    for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                        if (!mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitLimitNs)) {
                            record_failure(kRoleMma, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * S::kStageBytes);
                        const uint64_t a_desc = p.a_mn ? smem_desc_mnmajor_sw128(a_addr, kMnBoxBytes)
                                                       : smem_desc_kmajor_sw128(a_addr);
                        const uint64_t b_desc =
                            p.b_mn ? smem_desc_mnmajor_sw128(a_addr + S::kABytes, kMnBoxBytes)
                                   : smem_desc_kmajor_sw128(a_addr + S::kABytes);
#pragma unroll
                        for (int k = 0; k < BK / UK; ++k) {
                            tc_mma<kFmt>(d_tmem, a_desc + a_step * k, b_desc + b_step * k, idesc,
                                       (kb > kb_begin || k > 0) ? 1u : 0u);
                        }
                        tc_commit(&empty[stage]);
                        if (++stage == kStages) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit(&acc_full[acc]);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                }
            }
            // Every MMA issued so far must finish before TMEM is freed.
            tc_commit(drain);
            volatile int never = 0;
            mbar_wait_bounded(drain, 0, &never, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        const int ew = warp - 2;              // 0 .. kEpiWarps-1
        const int quarter = warp & 3;         // TMEM lanes this warp may access
        // INT8: four warps per lane quarter, each owning a quarter of the columns
        const int col_half = kI8 ? (ew >> 2) : 0;
        constexpr int kColsPerWarp = kI8 ? BN / 4 : BN;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t* stage =
            reinterpret_cast<uint32_t*>(smem + S::kEpiOffset + (ew & 7) * S::kEpiWarpBytes);
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (uint32_t t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
            uint32_t tm, tn;
            tile_coords(t, p, tm, tn);
            const int64_t row_base = static_cast<int64_t>(tm) * BM + quarter * 32;
            const int64_t col0 = static_cast<int64_t>(tn) * BN + col_half * kColsPerWarp;
            if constexpr (!kI8) {
                if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
                    record_failure(kRoleEpilogue, abort_flag);
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kColsPerWarp / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem_base + lane_base + acc * BN + c * 32, r);
                    tmem_ld_wait();
                    store_block_staged<TOut>(p, stage, lane, row_base, col0 + c * 32, r);
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            } else {
                int32_t sum[kColsPerWarp];
#pragma unroll
                for (int j = 0; j < kColsPerWarp; ++j) sum[j] = 0;
                const uint32_t n_chunks = (p.num_kb + kI8ChunkBlocks - 1) / kI8ChunkBlocks;
                for (uint32_t ch = 0; ch < n_chunks; ++ch) {
                    if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
                        record_failure(kRoleEpilogue, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // 16 columns per load: the 64 running sums and one load's
                    // registers stay within the 96 registers a thread of this
                    // 576-thread CTA has (32-column loads spilled)
#pragma unroll
                    for (int c = 0; c < kColsPerWarp / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(
                            tmem_base + lane_base + acc * BN + col_half * kColsPerWarp + c * 16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            // exact integer in fp32 (|x| <= 2^24) -> int32, wrapping add
                            sum[c * 16 + j] = static_cast<int32_t>(
                                static_cast<uint32_t>(sum[c * 16 + j]) +
                                static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j]))));
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&acc_empty[acc]);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                }
                if (!ok) break;
                // 16 warps, 8 staging squares: warps 0-7 store first, then 8-15
                // (named barrier 1 over the 512 epilogue threads).
                for (int round = 0; round < 2; ++round) {
                    if ((ew >> 3) == round) {
#pragma unroll
                        for (int c = 0; c < kColsPerWarp / 32; ++c)
                            store_block_staged_i32(p, stage, lane, row_base, col0 + c * 32,
                                                   &sum[c * 32]);
                    }
                    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---- the CTA-pair kernel (floating point) ---------------------------------------
//
// A cluster of two CTAs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): CTA r (r = 0, 1) loads
// rows [128r, 128r + 128) of the tile's A panel and rows [128r, 128r + 128) of
// its B panel (half of N) into its own shared memory, and its TMEM receives
// rows [128r, 128r + 128) of the accumulator (all 256 columns).  Compared with
// one CTA per 128 x 256 tile, each SM loads half as much B per MMA, so the
// same 192 KB ring holds 6 stages instead of 4.
//
// Roles and barriers (the even CTA is the leader):
//   * each CTA's TMA warp loads into its own ring; every copy counts its
//     bytes on the LEADER's full[s] barrier (cta_group::2 bulk tensor copy),
//     and the leader's producer announces the bytes of both CTAs;
//   * the leader's MMA thread issues the pair MMAs and commits, multicast to
//     both CTAs, to empty[s] (ring slot free) and acc_full[b] (accumulator
//     ready);
//   * each CTA's four epilogue warps drain their own TMEM and arrive (one lane
//     per warp) on the leader's acc_empty[b], which counts all eight warps.

constexpr int kPairStages = 6;
constexpr int kPairBN = 256;

// A 32 x 32 block of raw fp32 sums (as their bits) into a split tile's
// partial slot (256 x 256 words, row-major, tile-relative; rows and columns
// past the matrix are written too and never read), transposed through the
// staging square like the stores above.
__device__ __forceinline__ void store_block_partial(uint32_t* slot_base, uint32_t* stage, int lane,
                                                    int row_base, int col_base, const uint32_t* v) {
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = v[j];
    __syncwarp();
#pragma unroll 4
    for (int i = 0; i < 32; ++i)
        slot_base[(row_base + i) * kPairBN + col_base + lane] = stage[i * 33 + lane];
    __syncwarp();
}

// kSquares: epilogue staging squares, 4 for floating point (one per epilogue
// warp), 8 for INT8 (16 epilogue warps store in two rounds).
template <int kSquares>
struct PairSmem {
    static constexpr uint32_t kABytes = 128 * BK * 2;
    static constexpr uint32_t kBBytes = (kPairBN / 2) * BK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kRing = kPairStages * kStageBytes;
    static constexpr uint32_t kBarOffset = kRing;
    // full[S], empty[S], acc_full[2], acc_empty[2], drain, then tmem slot + abort flag
    static constexpr uint32_t kBarBytes = (2 * kPairStages + 5) * 8 + 16;
    static constexpr uint32_t kEpiOffset = (kBarOffset + kBarBytes + 127) / 128 * 128;
    static constexpr uint32_t kEpiWarpBytes = 32 * 33 * 4;
    static constexpr uint32_t kTotal = kEpiOffset + kSquares * kEpiWarpBytes;
    static constexpr uint32_t kLaunchBytes = kTotal + 1024;
};

template <uint32_t kFmt, bool kI8, typename TOut>
__global__ void __launch_bounds__(kI8 ? 576 : 192, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, TcParams p) {
    constexpr int kEpiWarps = kI8 ? 16 : 4;
    using S = PairSmem<kI8 ? 8 : 4>;
    constexpr uint32_t kTmemCols = 2 * kPairBN;  // two accumulators
    constexpr uint32_t kIdesc = idesc_mma(kFmt, 256, kPairBN);
    constexpr int kKElems = k_per_stage(kFmt);
    constexpr uint16_t kBothCtas = 0x3;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
    uint64_t* empty = full + kPairStages;
    uint64_t* acc_full = empty + kPairStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            // floating point: one lane of each epilogue warp of both CTAs;
            // INT8: one thread per CTA, after its 16 epilogue warps meet
            mbar_init(&acc_empty[b], kI8 ? 2 : 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // barriers of both CTAs initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // see the single-CTA kernel: the repack's output is read only after this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t cluster_id = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (uint32_t u = cluster_id; ok && u < p.num_units; u += n_clusters) {
                uint32_t tm, tn, kb_begin, kb_end;
                int32_t slot;
                unit_coords(u, p, tm, tn, kb_begin, kb_end, slot);
                const int32_t a_row = static_cast<int32_t>(tm * 256 + rank * 128);
                const int32_t b_row = static_cast<int32_t>(tn * kPairBN + rank * (kPairBN / 2));
                for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait_bounded<true>(&empty[stage], phase ^ 1, abort_flag,
                                                 kWaitLimitNs)) {
                        record_failure(kRoleProducer, abort_flag);
                        ok = false;
                        break;
                    }
                    uint8_t* a_dst = smem + stage * S::kStageBytes;
                    uint8_t* b_dst = a_dst + S::kABytes;
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * S::kStageBytes);
                    const uint32_t bar = map_to_cta(smem_u32(&full[stage]), 0);
                    const int32_t k0 = static_cast<int32_t>(kb * kKElems);
                    if (p.a_mn) {
                        for (uint32_t j = 0; j < BM / kMnAtom; ++j)
                            tma_load_2d_pair(a_dst + j * kMnBoxBytes, &tmA, bar,
                                             a_row + static_cast<int32_t>(j * kMnAtom), k0);
                    } else {
                        tma_load_2d_pair(a_dst, &tmA, bar, k0, a_row);
                    }
                    if (p.b_mn) {
                        for (uint32_t j = 0; j < (kPairBN / 2) / kMnAtom; ++j)
                            tma_load_2d_pair(b_dst + j * kMnBoxBytes, &tmB, bar,
                                             b_row + static_cast<int32_t>(j * kMnAtom), k0);
                    } else {
                        tma_load_2d_pair(b_dst, &tmB, bar, k0, b_row);
                    }
                    if (++stage == kPairStages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) __nanosleep(20000);  // let copies already issued land before teardown
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            const uint32_t idesc = idesc_major(kIdesc, p.a_mn, p.b_mn);
            const uint32_t a_step = p.a_mn ? kStepMnMajor : kStepKMajor;
            const uint32_t b_step = p.b_mn ? kStepMnMajor : kStepKMajor;
            bool ok = true;
            // INT8: the K loop of a tile is cut into exact 1024-deep chunks, each
            // in its own accumulator (see the single-CTA kernel); otherwise one
            // chunk spans the whole K loop
            for (uint32_t u = cluster_id; ok && u < p.num_units; u += n_clusters) {
                uint32_t tm, tn, kb_first, kb_last;
                int32_t slot;
                unit_coords(u, p, tm, tn, kb_first, kb_last, slot);
                const uint32_t n_chunks =
                    kI8 ? (kb_last - kb_first + kI8ChunkBlocks - 1) / kI8ChunkBlocks : 1;
                for (uint32_t ch = 0; ok && ch < n_chunks; ++ch) {
                    if (!mbar_wait_bounded<true>(&acc_empty[acc], acc_phase ^ 1, abort_flag,
                                                 kWaitLimitNs)) {
                        record_failure(kRoleMma, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * kPairBN;
                    const uint32_t kb_begin = kI8 ? kb_first + ch * kI8ChunkBlocks : kb_first;
                    const uint32_t kb_end = kI8 ? min(kb_last, kb_begin + kI8ChunkBlocks) : kb_last;
                    for (uint32_t kb = kb_begin; kb < kb_end; ++kb) {
                        if (!mbar_wait_bounded<true>(&full[stage], phase, abort_flag, kWaitLimitNs)) {
                            record_failure(kRoleMma, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * S::kStageBytes);
                        const uint64_t a_desc = p.a_mn ? smem_desc_mnmajor_sw128(a_addr, kMnBoxBytes)
                                                       : smem_desc_kmajor_sw128(a_addr);
                        const uint64_t b_desc =
                            p.b_mn ? smem_desc_mnmajor_sw128(a_addr + S::kABytes, kMnBoxBytes)
                                   : smem_desc_kmajor_sw128(a_addr + S::kABytes);
#pragma unroll
                        for (int k = 0; k < BK / UK; ++k)
                            tc_mma_pair<kFmt>(d_tmem, a_desc + a_step * k, b_desc + b_step * k,
                                              idesc, (kb > kb_begin || k > 0) ? 1u : 0u);
                        tc_commit_pair_multicast(&empty[stage], kBothCtas);
                        if (++stage == kPairStages) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit_pair_multicast(&acc_full[acc], kBothCtas);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                }
            }
            // every pair MMA issued so far must finish before TMEM is freed
            tc_commit_pair_multicast(drain, 0x1);
            volatile int never = 0;
            mbar_wait_bounded(drain, 0, &never, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue warps (both CTAs)
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t* stage =
            reinterpret_cast<uint32_t*>(smem + S::kEpiOffset + (ew & 7) * S::kEpiWarpBytes);
        // INT8: four warps per lane quarter, each owning a quarter of the columns
        const int col_group = kI8 ? (ew >> 2) : 0;
        constexpr int kColsPerWarp = kI8 ? kPairBN / 4 : kPairBN;
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (uint32_t u = cluster_id; ok && u < p.num_units; u += n_clusters) {
            // INT8 never splits (each unit a whole tile): its 64 running sums
            // leave no registers for a unit's k-range, and a split measured
            // slower (the parts' epilogues cost more than the shorter wave)
            uint32_t tm, tn, kb_first = 0, kb_last = p.num_kb;
            int32_t slot = -1;
            if constexpr (kI8) tile_coords(u, p, tm, tn);
            else unit_coords(u, p, tm, tn, kb_first, kb_last, slot);
            const int64_t row_base = static_cast<int64_t>(tm) * 256 + rank * 128 + quarter * 32;
            const int64_t col0 = static_cast<int64_t>(tn) * kPairBN + col_group * kColsPerWarp;
            if constexpr (!kI8) {
                if (!mbar_wait_bounded<true>(&acc_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
                    record_failure(kRoleEpilogue, abort_flag);
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kPairBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem_base + lane_base + acc * kPairBN + c * 32, r);
                    tmem_ld_wait();
                    if (slot < 0)
                        store_block_staged<TOut>(p, stage, lane, row_base, col0 + c * 32, r);
                    else
                        store_block_partial(p.partials + static_cast<int64_t>(slot) * (256 * kPairBN),
                                            stage, lane, static_cast<int>(rank * 128 + quarter * 32),
                                            c * 32, r);  // r: the fp32 sums' bits
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&acc_empty[acc]), 0));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            } else {
                // each chunk's exact fp32 sums become int32 and add up (wrapping)
                int32_t sum[kColsPerWarp];
#pragma unroll
                for (int j = 0; j < kColsPerWarp; ++j) sum[j] = 0;
                const uint32_t n_chunks = (p.num_kb + kI8ChunkBlocks - 1) / kI8ChunkBlocks;
                for (uint32_t ch = 0; ch < n_chunks; ++ch) {
                    if (!mbar_wait_bounded<true>(&acc_full[acc], acc_phase, abort_flag,
                                                 kWaitLimitNs)) {
                        record_failure(kRoleEpilogue, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // 16 columns per load (see the single-CTA kernel: no spills)
#pragma unroll
                    for (int c = 0; c < kColsPerWarp / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(tmem_base + lane_base + acc * kPairBN +
                                               col_group * kColsPerWarp + c * 16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            sum[c * 16 + j] = static_cast<int32_t>(
                                static_cast<uint32_t>(sum[c * 16 + j]) +
                                static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j]))));
                    }
                    // every epilogue warp of this CTA has read the accumulator: one
                    // thread tells the leader (a single cluster-scope release per CTA)
                    tc_fence_before();
                    asm volatile("bar.sync 2, %0;" ::"n"(kEpiWarps * 32) : "memory");
                    if (ew == 0 && lane == 0)
                        mbar_arrive_cluster(map_to_cta(smem_u32(&acc_empty[acc]), 0));
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                }
                if (!ok) break;
                // 16 warps, 8 staging squares: warps 0-7 store first, then 8-15
                // (named barrier 1 over this CTA's 512 epilogue threads)
                for (int round = 0; round < 2; ++round) {
                    if ((ew >> 3) == round) {
#pragma unroll
                        for (int c = 0; c < kColsPerWarp / 32; ++c)
                            store_block_staged_i32(p, stage, lane, row_base, col0 + c * 32,
                                                   &sum[c * 32]);
                    }
                    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // no CTA frees TMEM or exits while its peer may still touch it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// ---- the split last wave's reduce ------------------------------------------------
//
// Adds the K-parts of each split tile (full_tiles + j) in part order, i.e. in
// K order, so that the result repeats bit for bit, and applies the epilogue
// as store_block_staged does (alpha, beta -- C is read only when beta != 0 --
// the bias row, the edge masks, the output type).  One block per 8 rows of a
// tile, a warp per row, lane l taking columns l, l + 32, ..., l + 224: every
// load and store instruction covers 32 consecutive elements.  Launched as a
// programmatic dependent of the GEMM: it reads the partial sums only after
// griddepcontrol.wait.
template <typename TOut>
__global__ void __launch_bounds__(256) tc_split_reduce_kernel(TcParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t j = blockIdx.x / 32;
    const int r = static_cast<int>(blockIdx.x % 32) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    uint32_t tm, tn;
    tile_coords(p.full_tiles + j, p, tm, tn);
    const int64_t row = static_cast<int64_t>(tm) * 256 + r;
    if (row >= p.M) return;
    constexpr int64_t kSlot = 256 * kPairBN;
    const float* base = reinterpret_cast<const float*>(p.partials) +
                        static_cast<int64_t>(j) * p.splits * kSlot + r * kPairBN + lane;
    float sum[kPairBN / 32];
#pragma unroll
    for (int q = 0; q < kPairBN / 32; ++q) sum[q] = base[q * 32];
    for (uint32_t part = 1; part < p.splits; ++part) {
        const float* b = base + part * kSlot;
        float v[kPairBN / 32];
#pragma unroll
        for (int q = 0; q < kPairBN / 32; ++q) v[q] = b[q * 32];
#pragma unroll
        for (int q = 0; q < kPairBN / 32; ++q) sum[q] += v[q];
    }
#pragma unroll
    for (int q = 0; q < kPairBN / 32; ++q) {
        const int64_t col = static_cast<int64_t>(tn) * kPairBN + q * 32 + lane;
        if (col < p.N) {
            TOut* dst = static_cast<TOut*>(p.C) + row * p.ldc + col;
            const float old = p.beta != 0.0f ? OutT<TOut>::load(dst) : 0.0f;
            const float bv = p.bias != nullptr ? OutT<TOut>::load(static_cast<const TOut*>(p.bias) + col) : 0.0f;
            OutT<TOut>::store(dst, axpby(p.alpha, sum[q], p.beta, old) + bv);
        }
    }
}

// ---- self-test of the bounded wait ----------------------------------------------
//
// Waits on an mbarrier that nothing ever arrives at, with the same bounded
// wait the GEMM roles use, so that the give-up path (status word, abort
// flag, orderly return) can be exercised on a GPU without hanging it.

__global__ void bounded_wait_probe_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int* flag = &abort_flag;
        if (!mbar_wait_bounded(&bar, 0, flag, limit_ns)) record_failure(kRoleSelfTest, flag);
    }
}

// ---- operand repacking into the workspace ------------------------------------
//
// 16-bit operands: dst[r][c] = src[r*ld_src + c] converted to 16-bit storage
// (bf16/fp16; int8 values become exact bf16), for r < rows, c < the row
// length, and zero up to ld_dst, a multiple of 8 (every thread writes whole
// 16-byte vectors).  The rows are the source's own: K-long rows of a K-major
// operand, M- or N-long rows (one per k) of an MN-major one, which the GEMM
// then reads MN-major.  fp32 operands of the TF32 path (K-major only) are
// copied, or transposed, by their own kernels.

template <typename TSrc> struct PackIn;  // 16-bit sources: their bits
template <> struct PackIn<__nv_bfloat16> {
    __device__ __forceinline__ static uint16_t bits(__nv_bfloat16 v) { return __bfloat16_as_ushort(v); }
};
template <> struct PackIn<__half> {
    __device__ __forceinline__ static uint16_t bits(__half v) { return __half_as_ushort(v); }
};

__device__ __forceinline__ uint4 pack8(const uint16_t (&h)[8]) {
    return make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                      h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
}

// One operand's repack, as the fused kernel below receives it: dst[r][k] =
// src[r*ld_src + k] converted, for r < rows, k < K (the row length: K for a
// K-major operand, M or N for an MN-major one), zero for K <= k < ld_dst.
template <typename TSrc>
struct PackJob {
    const TSrc* src;
    const TSrc* src_end;  // one past the last element of the last row
    int64_t ld_src, rows, K;
    uint16_t* dst;
    int64_t ld_dst;
    int vec_src;      // the source's 8-element groups are aligned
    int64_t blocks;   // blocks of the launch this job takes
    // the unit of work: 8 elements of a row per thread (16-bit sources) or
    // 1024 elements of a row per warp (int8); units_per_row = ld_dst / unit,
    // rounded up
    int64_t units_per_row;
    // unit index i -> row i / units_per_row as (i * div_m) >> div_s, exact
    // for i < 2^31 (a precomputed reciprocal: no division in the kernel);
    // used when fast_div, i.e. when the job has fewer than 2^31 units
    uint64_t div_m;
    int div_s, fast_div;
    // int8 only: the source is the operand's transpose, element (k, r) at
    // src[k*ld_src + r] for k < K, r < rows, and the copy transposes it in
    // 64 (k) x 128 (r) tiles, tiles_k of them along each 128 rows
    int transpose;
    int64_t tiles_k;
};

// Eight int8 values (byte q of v is value q) as eight exact bf16, in memory
// order, without conversion instructions (those issue at a fraction of the
// integer and FMA rate): for a byte b, u = b ^ 0x80 is v + 128, and the float
// whose bits are 0x4B000000 | u is exactly 2^23 + u, so subtracting
// 2^23 + 128 gives v exactly (one FADD); an integer of magnitude <= 128 has at
// most 8 significant bits, so the top 16 bits of its float encoding are its
// bf16 encoding, and one byte permute packs two of them.
__device__ __forceinline__ uint4 int8x8_to_bf16(uint64_t v) {
    const uint32_t w[2] = {static_cast<uint32_t>(v) ^ 0x80808080u,
                           static_cast<uint32_t>(v >> 32) ^ 0x80808080u};
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t x = w[q >> 1];
        const uint32_t b0 = (2 * q) & 3, b1 = (2 * q + 1) & 3;  // byte positions in x
        // bytes of the result: [x byte b, 0x00, 0x00, 0x4B] (selector digits 4 and 7 pick
        // bytes 0 and 3 of the constant)
        const float f0 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | b0)) - 8388736.0f;
        const float f1 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | b1)) - 8388736.0f;
        out[q] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);  // top halves
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint64_t ldg_u64(uintptr_t a) {
    return __ldg(reinterpret_cast<const unsigned long long*>(a));
}

// The row of a job's unit i (units_per_row units per row): i / units_per_row
// through the job's precomputed reciprocal where it is exact.
template <typename TSrc>
__device__ __forceinline__ int64_t unit_row(const PackJob<TSrc>& j, int64_t i) {
    if (j.fast_div) return static_cast<int64_t>((static_cast<uint64_t>(i) * j.div_m) >> j.div_s);
    return i / j.units_per_row;
}

// 16-bit sources: one thread per 8 consecutive elements of a row (block-stride
// over `nblocks` blocks, this one being `blk`), copied bit for bit.
template <typename TSrc>
__device__ __forceinline__ void pack_rows_body(const PackJob<TSrc>& j, int64_t blk, int64_t nblocks) {
    const TSrc* __restrict__ src = j.src;
    uint16_t* __restrict__ dst = j.dst;
    const int64_t ld_src = j.ld_src, K = j.K, ld_dst = j.ld_dst;
    const int64_t total = j.rows * j.units_per_row;
    for (int64_t i = blk * 256 + threadIdx.x; i < total; i += nblocks * 256) {
        const int64_t r = unit_row(j, i), k = (i - r * j.units_per_row) * 8;
        const TSrc* s = src + r * ld_src + k;
        uint16_t h[8];
        if (j.vec_src && k + 8 <= K) {
            TSrc v[8];
            *reinterpret_cast<uint4*>(v) = __ldg(reinterpret_cast<const uint4*>(s));
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = PackIn<TSrc>::bits(v[q]);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = k + q < K ? PackIn<TSrc>::bits(s[q]) : uint16_t(0);
        }
        *reinterpret_cast<uint4*>(dst + r * ld_dst + k) = pack8(h);
    }
}

// int8 sources: a warp's unit is 128 consecutive output vectors (8 bf16 each)
// of one row, lane l taking vectors l, l + 32, l + 64 and l + 96, so every
// warp-wide load reads 256 contiguous bytes and every warp-wide store writes
// 512.  A vector's 8 source bytes are one aligned 64-bit word for a row that
// is 8-byte aligned, else the two aligned words around them, funnel-shifted
// (only where both lie inside the operand: [src, src_end)); bytewise at the
// row's end and at the operand's edges.  All four vectors' loads are issued
// before the first conversion.
template <>
__device__ __forceinline__ void pack_rows_body<int8_t>(const PackJob<int8_t>& j, int64_t blk,
                                                       int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t vec_per_row = j.ld_dst / 8;
    const int64_t total = j.rows * j.units_per_row;  // warp units
    const uintptr_t lo = reinterpret_cast<uintptr_t>(j.src), hi = reinterpret_cast<uintptr_t>(j.src_end);
    for (int64_t wu = blk * 8 + (threadIdx.x >> 5); wu < total; wu += nblocks * 8) {
        const int64_t r = unit_row(j, wu), seg = wu - r * j.units_per_row;
        const int8_t* row = j.src + r * j.ld_src;
        uint64_t w[4];
        // a unit whose 1024 elements all lie in the row (and, for unaligned
        // rows, whose word pairs all lie in the operand) loads without checks
        const int8_t* p = row + seg * 1024 + 8 * lane;
        const uintptr_t ulast = reinterpret_cast<uintptr_t>(row + seg * 1024 + 1016);
        const bool whole = seg * 1024 + 1024 <= j.K &&
                           (j.vec_src || ((reinterpret_cast<uintptr_t>(row + seg * 1024) & ~static_cast<uintptr_t>(7)) >= lo &&
                                          (ulast & ~static_cast<uintptr_t>(7)) + 16 <= hi));
        if (whole) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(p + 256 * q);
                if (j.vec_src) {
                    w[q] = ldg_u64(a);
                } else {
                    const uintptr_t base = a & ~static_cast<uintptr_t>(7);
                    const uint64_t x0 = ldg_u64(base), x1 = ldg_u64(base + 8);
                    const int sh = static_cast<int>(a - base) * 8;
                    w[q] = sh ? (x0 >> sh) | (x1 << (64 - sh)) : x0;
                }
            }
            uint16_t* d = j.dst + r * j.ld_dst + seg * 1024 + 8 * lane;
#pragma unroll
            for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(d + 256 * q) = int8x8_to_bf16(w[q]);
            continue;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t v = seg * 128 + lane + 32 * q;
            const int64_t k = 8 * v;
            w[q] = 0;
            if (v >= vec_per_row) continue;
            const uintptr_t a = reinterpret_cast<uintptr_t>(row + k);
            bool have = false;
            if (k + 8 <= j.K) {
                if (j.vec_src) {
                    w[q] = ldg_u64(a);
                    have = true;
                } else {
                    const uintptr_t base = a & ~static_cast<uintptr_t>(7);
                    if (base >= lo && base + 16 <= hi) {
                        const uint64_t x0 = ldg_u64(base), x1 = ldg_u64(base + 8);
                        const int sh = static_cast<int>(a - base) * 8;
                        w[q] = sh ? (x0 >> sh) | (x1 << (64 - sh)) : x0;
                        have = true;
                    }
                }
            }
            if (!have) {
                for (int b = 0; b < 8; ++b)
                    if (k + b < j.K) w[q] |= static_cast<uint64_t>(static_cast<uint8_t>(row[k + b])) << (8 * b);
            }
        }
        uint16_t* d = j.dst + r * j.ld_dst;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t v = seg * 128 + lane + 32 * q;
            if (v < vec_per_row) *reinterpret_cast<uint4*>(d + 8 * v) = int8x8_to_bf16(w[q]);
        }
    }
}

// The 8 source bytes (k, r .. r + 7) of a transposing int8 job, zero past
// the source's extent: one aligned word where rows are 8-byte aligned, else
// the two aligned words around them funnel-shifted (only where both lie in
// [src, src_end)), else byte by byte.
__device__ __forceinline__ uint64_t load_i8x8(const PackJob<int8_t>& j, int64_t k, int64_t r) {
    if (k >= j.K || r >= j.rows) return 0;
    const int8_t* p = j.src + k * j.ld_src + r;
    if (r + 8 <= j.rows) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        if (j.vec_src) return ldg_u64(a);
        const uintptr_t base = a & ~static_cast<uintptr_t>(7);
        if (base >= reinterpret_cast<uintptr_t>(j.src) &&
            base + 16 <= reinterpret_cast<uintptr_t>(j.src_end)) {
            const uint64_t x0 = ldg_u64(base), x1 = ldg_u64(base + 8);
            const int sh = static_cast<int>(a - base) * 8;
            return sh ? (x0 >> sh) | (x1 << (64 - sh)) : x0;
        }
    }
    uint64_t w = 0;
    for (int b = 0; b < 8 && r + b < j.rows; ++b)
        w |= static_cast<uint64_t>(static_cast<uint8_t>(p[b])) << (8 * b);
    return w;
}

// Transposing int8 job: dst[r][k] = src[k*ld_src + r] as bf16, a 64 (k) x
// 128 (r) tile per block at a time.  Thread t loads the 8 source bytes at
// r = 8*(t % 16) of the 4 rows k = 4*(t / 16) .. + 3 (a warp reads 2 x 128
// contiguous bytes per load), regroups them with byte permutes into 8 words
// of 4 consecutive k, one per r, and stores them to a shared tile of 128 rows
// x 16 words, word kq of row r at kq ^ h(r), h(r) = ((r >> 1) & 1) |
// (((r >> 3) & 7) << 1): the stores hit 16 banks per instruction (every
// lane's row has the same parity, so 16 is the most a row stride of 64 bytes
// allows) and the reads below all 32.  A warp then converts and writes whole
// 128-byte output segments, 4 rows x 8 vectors of 8 k per instruction.
__device__ __forceinline__ void pack_tiles_i8_body(const PackJob<int8_t>& j, int64_t blk,
                                                   int64_t nblocks, uint32_t* tile) {
    const int t = threadIdx.x;
    const int64_t tiles = ((j.rows + 127) / 128) * j.tiles_k;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(j.src), hi = reinterpret_cast<uintptr_t>(j.src_end);
    for (int64_t i = blk; i < tiles; i += nblocks) {
        const int64_t tr = unit_row(j, i), tk = i - tr * j.tiles_k;
        const int64_t r0 = tr * 128, k0 = tk * 64;
        const int wn = t & 15, kq = t >> 4;
        // an interior tile (all 64 x 128 bytes inside the operand, and for
        // unaligned rows every word pair around them too) loads without checks
        const uintptr_t first = reinterpret_cast<uintptr_t>(j.src + k0 * j.ld_src + r0);
        const uintptr_t last = reinterpret_cast<uintptr_t>(j.src + (k0 + 63) * j.ld_src + r0 + 120);
        const bool interior = k0 + 64 <= j.K && r0 + 128 <= j.rows &&
                              (j.vec_src || ((first & ~static_cast<uintptr_t>(7)) >= lo &&
                                             (last & ~static_cast<uintptr_t>(7)) + 16 <= hi));
        uint64_t w[4];
        if (interior) {
            const int8_t* p = j.src + (k0 + 4 * kq) * j.ld_src + r0 + 8 * wn;
            if (j.vec_src) {
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = ldg_u64(reinterpret_cast<uintptr_t>(p + q * j.ld_src));
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uintptr_t a = reinterpret_cast<uintptr_t>(p + q * j.ld_src);
                    const uintptr_t base = a & ~static_cast<uintptr_t>(7);
                    const uint64_t x0 = ldg_u64(base), x1 = ldg_u64(base + 8);
                    const int sh = static_cast<int>(a - base) * 8;
                    w[q] = sh ? (x0 >> sh) | (x1 << (64 - sh)) : x0;
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = load_i8x8(j, k0 + 4 * kq + q, r0 + 8 * wn);
        }
        // column c of the 4 x 8 byte block: bytes (k0 + 4kq + 0..3, r0 + 8wn + c)
        uint32_t col[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t x0 = static_cast<uint32_t>(w[0] >> (32 * h));
            const uint32_t x1 = static_cast<uint32_t>(w[1] >> (32 * h));
            const uint32_t x2 = static_cast<uint32_t>(w[2] >> (32 * h));
            const uint32_t x3 = static_cast<uint32_t>(w[3] >> (32 * h));
            const uint32_t p01 = __byte_perm(x0, x1, 0x5140), q01 = __byte_perm(x0, x1, 0x7362);
            const uint32_t p23 = __byte_perm(x2, x3, 0x5140), q23 = __byte_perm(x2, x3, 0x7362);
            col[4 * h + 0] = __byte_perm(p01, p23, 0x5410);
            col[4 * h + 1] = __byte_perm(p01, p23, 0x7632);
            col[4 * h + 2] = __byte_perm(q01, q23, 0x5410);
            col[4 * h + 3] = __byte_perm(q01, q23, 0x7632);
        }
        __syncthreads();  // the previous tile's reads are done
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int r = 8 * wn + c;
            const int hr = ((r >> 1) & 1) | (((r >> 3) & 7) << 1);
            tile[r * 16 + (kq ^ hr)] = col[c];
        }
        __syncthreads();
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 32 + (t >> 3), g = t & 7;
            const int hr = ((r >> 1) & 1) | (((r >> 3) & 7) << 1);
            // words 2g and 2g + 1 sit together at 2 (g ^ (hr >> 1)), swapped when hr is odd
            const uint2 v = *reinterpret_cast<const uint2*>(tile + r * 16 + 2 * (g ^ (hr >> 1)));
            const uint32_t k_lo = (hr & 1) ? v.y : v.x, k_hi = (hr & 1) ? v.x : v.y;
            const int64_t row = r0 + r, k = k0 + 8 * g;
            if (row < j.rows && k < j.ld_dst)
                *reinterpret_cast<uint4*>(j.dst + row * j.ld_dst + k) =
                    int8x8_to_bf16(static_cast<uint64_t>(k_lo) | (static_cast<uint64_t>(k_hi) << 32));
        }
    }
}

// Both operands' repacks in one launch: blocks [0, a.blocks) do A's job, the
// rest B's (a job with 0 blocks is absent).  A 16-bit repack copies its
// source row by row, keeping the layout (an MN-major operand stays MN-major);
// an int8 one re-encodes as bf16 and leaves both operands K-major, copying
// row-major A and column-major B by rows and transposing column-major A and
// row-major B by tiles.  One launch lets B's blocks fill the SMs while A's
// drain, and the GEMM behind it is released (griddepcontrol.launch_dependents)
// as soon as every block has started: its prologue overlaps the repack's
// tail, and it reads the output only after griddepcontrol.wait, i.e. after
// this grid has completed.
template <typename TSrc>
__device__ __forceinline__ void pack_job_body(const PackJob<TSrc>& j, int64_t blk, uint32_t* tile) {
    if constexpr (sizeof(TSrc) == 1) {
        if (j.transpose) {
            pack_tiles_i8_body(j, blk, j.blocks, tile);
            return;
        }
    }
    pack_rows_body(j, blk, j.blocks);
}

template <typename TSrc>
__global__ void __launch_bounds__(256) pack_pair_kernel(PackJob<TSrc> a, PackJob<TSrc> b) {
    // the transposing int8 tiles' staging (unused by 16-bit repacks)
    __shared__ __align__(16) uint32_t tile[sizeof(TSrc) == 1 ? 128 * 16 : 1];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t blk = blockIdx.x;
    if (blk < a.blocks) pack_job_body(a, blk, tile);
    else pack_job_body(b, blk - a.blocks, tile);
}

// fp32 operands of the TF32 path, same contract with 4-byte elements:
// dst[r][k] = src(r, k) for k < K, zero for K <= k < ld_dst (ld_dst % 4 == 0,
// so every thread writes whole 16-byte vectors).
__global__ void __launch_bounds__(256) pack_rows_f32_kernel(const float* __restrict__ src,
                                                            int64_t ld_src, int64_t rows, int64_t K,
                                                            float* __restrict__ dst, int64_t ld_dst) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // see pack_pair_kernel
    const int64_t groups = ld_dst / 4;
    const int64_t total = rows * groups;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / groups, k = (i % groups) * 4;
        const float* s = src + r * ld_src + k;
        float4 v;
        v.x = k < K ? s[0] : 0.0f;
        v.y = k + 1 < K ? s[1] : 0.0f;
        v.z = k + 2 < K ? s[2] : 0.0f;
        v.w = k + 3 < K ? s[3] : 0.0f;
        *reinterpret_cast<float4*>(dst + r * ld_dst + k) = v;
    }
}

// Transposed fp32 source, src(r, k) = src[k*ld_src + r]: a 64 (k) x 64 (r)
// tile per block through shared memory; reads walk r, writes walk k.
__global__ void __launch_bounds__(256) pack_transposed_f32_kernel(const float* __restrict__ src,
                                                                  int64_t ld_src, int64_t rows,
                                                                  int64_t K, float* __restrict__ dst,
                                                                  int64_t ld_dst) {
    __shared__ float tile[64][64 + 1];  // tile[k][r]
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // see pack_pair_kernel
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64;
    const int t = threadIdx.x;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const int idx = i * 256 + t, kk = idx >> 6, rr = idx & 63;
        const int64_t k = k0 + kk, r = r0 + rr;
        tile[kk][rr] = (k < K && r < rows) ? src[k * ld_src + r] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = i * 256 + t, rr = idx >> 4, kq = (idx & 15) * 4;
        const int64_t r = r0 + rr, k = k0 + kq;
        if (r < rows && k < ld_dst)
            *reinterpret_cast<float4*>(dst + r * ld_dst + k) =
                make_float4(tile[kq][rr], tile[kq + 1][rr], tile[kq + 2][rr], tile[kq + 3][rr]);
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

// Tensor-map element type and size of an operand format.
CUtensorMapDataType map_dtype(uint32_t fmt) {
    return fmt == kFmtTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                           : (fmt == kFmtBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}
int64_t elem_bytes(uint32_t fmt) { return fmt == kFmtTF32 ? 4 : 2; }

// K-major operand: rows x K elements, row stride ld elements; boxes of one
// 128-byte row of K (64 16-bit or 32 fp32 elements) x box_rows.
cudaError_t make_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                            int64_t ld, uint32_t box_rows, uint32_t fmt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * elem_bytes(fmt))};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(k_per_stage(fmt)), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, map_dtype(fmt), 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// MN-major operand: MN x K elements of 2 bytes with MN contiguous, k-row
// stride ld elements; boxes of 64 MN-elements x 64 k.
cudaError_t make_mnmajor_map(CUtensorMap* map, const void* base, int64_t mn, int64_t K,
                             int64_t ld, uint32_t fmt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(mn), static_cast<cuuint64_t>(K)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {kMnAtom, static_cast<cuuint32_t>(BK)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, map_dtype(fmt), 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

constexpr int kBnFloat = 256;
constexpr int kBnI8 = 256;
constexpr size_t kWsAlign = 256;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Which operands need repacking into the workspace.  16-bit repacks keep the
// operand's own layout: a K-major operand becomes rows x kp, an MN-major one
// (column-major A, row-major B) K rows x ld_mn, both copied row by row.
struct PackPlan {
    bool pack_a, pack_b;
    bool a_mn, b_mn;  // read MN-major (column-major A / row-major B)
    int64_t kp;  // padded K of K-major repacks (multiple of 8 elements = 16 bytes)
    int64_t a_ld, b_ld;  // leading dimension of each repacked operand
    size_t a_bytes, b_bytes;
};

PackPlan plan_for(const GemmArgs& a) {
    PackPlan pl{};
    const bool i8 = a.in_dtype == DGA_I8;
    if (a.in_dtype == DGA_TF32) {
        // fp32 rows (4 elements = 16 bytes); TF32 operands are always K-major,
        // so a column-major A or row-major B is transposed into the workspace
        pl.kp = round_up(a.K, 4);
        pl.pack_a = a.layout_a == DGA_COL_MAJOR || a.lda % 4 != 0 || !aligned(a.A, 16);
        pl.pack_b = a.layout_b == DGA_ROW_MAJOR || a.ldb % 4 != 0 || !aligned(a.B, 16);
        pl.a_mn = pl.b_mn = false;
        pl.a_ld = pl.b_ld = pl.kp;
        pl.a_bytes = pl.pack_a ? round_up(a.M * pl.kp * 4, kWsAlign) : 0;
        pl.b_bytes = pl.pack_b ? round_up(a.N * pl.kp * 4, kWsAlign) : 0;
        return pl;
    }
    pl.kp = round_up(a.K, 8);
    // TMA needs 16-byte row strides and a 16-byte aligned base; INT8 is
    // always re-encoded (as bf16), into K-major rows whatever the source's
    // layout (the MMA reads a K-major B faster).  A 16-bit copy keeps the
    // layout: MN-major operands are read MN-major from it.
    pl.pack_a = i8 || a.lda % 8 != 0 || !aligned(a.A, 16);
    pl.pack_b = i8 || a.ldb % 8 != 0 || !aligned(a.B, 16);
    pl.a_mn = !i8 && a.layout_a == DGA_COL_MAJOR;
    pl.b_mn = !i8 && a.layout_b == DGA_ROW_MAJOR;
    pl.a_ld = pl.a_mn ? round_up(a.M, 8) : pl.kp;
    pl.b_ld = pl.b_mn ? round_up(a.N, 8) : pl.kp;
    pl.a_bytes = pl.pack_a ? round_up((pl.a_mn ? a.K : a.M) * pl.a_ld * 2, kWsAlign) : 0;
    pl.b_bytes = pl.pack_b ? round_up((pl.b_mn ? a.K : a.N) * pl.b_ld * 2, kWsAlign) : 0;
    return pl;
}

// Workspace size when pointers are not known: assume aligned pointers.
PackPlan plan_for_sizes(const GemmArgs& a) {
    GemmArgs b = a;
    static const char aligned_probe[16] __attribute__((aligned(16))) = {};
    b.A = aligned_probe;
    b.B = aligned_probe;
    return plan_for(b);
}

// Tile rows per raster group.  The resident CTAs work on consecutive tiles,
// i.e. on `group_m` tile rows at a time while B's column panels stream past;
// the A panels of one group should stay in L2 (half of it, leaving room for
// the streamed B panels and C), and the larger the group the fewer times B
// is read from DRAM.
uint32_t raster_group_rows(int64_t K, uint32_t tiles_m, int tile_rows) {
    const double a_panel = static_cast<double>(tile_rows) * K * 2;  // bytes of one A tile row
    const double budget = 32.0 * 1024 * 1024;  // measured best: 16 tile rows at K = 8192
    uint32_t g = static_cast<uint32_t>(budget / a_panel);
    g = std::max<uint32_t>(8, std::min<uint32_t>(g, 64));
    return std::min(g, tiles_m);
}

// pdl: the launch follows the operand repack on `s` and may start before it
// completes (programmatic stream serialisation; the kernel waits for it with
// griddepcontrol.wait before its first operand load).
template <uint32_t kFmt, bool kI8, int BN, typename TOut>
cudaError_t launch_kernel(const CUtensorMap& ma, const CUtensorMap& mb, const TcParams& p,
                          const DeviceInfo& dev, cudaStream_t s, bool pdl) {
    auto kern = tc_gemm_kernel<kFmt, kI8, BN, TOut>;
    const int smem = static_cast<int>(Smem<BN, kI8 ? 8 : 4>::kLaunchBytes);
    if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<uint32_t>(p.num_tiles, dev.sm_count)));
    cfg.blockDim = dim3(kI8 ? 576 : 192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, p);
}

// Clusters of two that fit at once on this device (queried once per kernel
// and device: the template arguments name the kernel, since every pair
// kernel has the same function type and would otherwise share one cache).
template <uint32_t kFmt, bool kI8, typename TOut, typename Kern>
int max_pair_clusters(Kern kern, int smem, int threads, const DeviceInfo& dev) {
    static int cached[64] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (dev.ordinal >= 0 && dev.ordinal < 64 && cached[dev.ordinal] > 0) return cached[dev.ordinal];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = dev.sm_count / 2;
    }
    if (dev.ordinal >= 0 && dev.ordinal < 64) cached[dev.ordinal] = n;
    return n;
}

// The split of the last wave: at most kMaxSplits parts per tile, none
// shallower than kMinSplitKb k-blocks, at most two rounds of parts (so at
// most 2 x clusters slots of workspace, 256 x 256 32-bit words each).
constexpr uint32_t kMaxSplits = 4;
constexpr uint32_t kMinSplitKb = 8;
constexpr size_t kSplitSlotBytes = size_t{256} * kPairBN * sizeof(uint32_t);

// Parts per tile for a last wave of `rem` tiles on `nc` clusters: the s that
// makes that wave shortest, ceil(rem * s / nc) rounds of 1/s of a tile time
// (the smaller s on a tie); 1 when no split shortens it.
uint32_t split_parts(uint32_t rem, uint32_t nc, uint32_t num_kb) {
    uint32_t best = 1, best_rounds = 1;  // one round of whole tiles
    const uint32_t s_max = std::min(kMaxSplits, num_kb / kMinSplitKb);
    for (uint32_t sp = 2; sp <= s_max; ++sp) {
        if (rem * sp > 2 * nc) break;
        const uint32_t rounds = (rem * sp + nc - 1) / nc;
        if (rounds * best < best_rounds * sp) {  // rounds / sp < best_rounds / best
            best = sp;
            best_rounds = rounds;
        }
    }
    return best;
}

// The CTA-pair GEMM, and for floating point, when split_ws holds enough and a
// split shortens the last, part-filled wave (split_parts), the split of that
// wave's tiles along K into work units of their own and the reduce that adds
// the parts (*extra_launches is incremented for it).
template <uint32_t kFmt, bool kI8, typename TOut>
cudaError_t launch_pair_kernel(const CUtensorMap& ma, const CUtensorMap& mb, const TcParams& p0,
                               const DeviceInfo& dev, cudaStream_t s, bool pdl, uint32_t* split_ws,
                               size_t split_bytes, int* extra_launches) {
    auto kern = tc_gemm_pair_kernel<kFmt, kI8, TOut>;
    const int smem = static_cast<int>(PairSmem<kI8 ? 8 : 4>::kLaunchBytes);
    const int threads = kI8 ? 576 : 192;
    if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int clusters = std::min<int64_t>(
        p0.num_tiles, max_pair_clusters<kFmt, kI8, TOut>(kern, smem, threads, dev));
    TcParams p = p0;
    p.full_tiles = p.num_tiles;
    p.splits = 1;
    p.num_units = p.num_tiles;
    p.partials = nullptr;
    const uint32_t nc = static_cast<uint32_t>(std::max(clusters, 1));
    if (!kI8 && split_ws != nullptr && p.num_tiles > nc) {
        const uint32_t rem = p.num_tiles % nc;
        const uint32_t sp = rem > 0 ? split_parts(rem, nc, p.num_kb) : 1;
        if (sp >= 2 && static_cast<size_t>(rem) * sp * kSplitSlotBytes <= split_bytes) {
            p.full_tiles = p.num_tiles - rem;
            p.splits = sp;
            p.num_units = p.full_tiles + rem * sp;
            p.partials = split_ws;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * std::max(clusters, 1)));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;  // see launch_kernel
    e = cudaLaunchKernelEx(&cfg, kern, ma, mb, p);
    if (e != cudaSuccess || p.splits == 1) return e;
    if constexpr (!kI8) {
        cudaLaunchConfig_t rc = {};
        rc.gridDim = dim3((p.num_tiles - p.full_tiles) * 32);
        rc.blockDim = dim3(256);
        rc.stream = s;
        cudaLaunchAttribute ra[1];
        ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ra[0].val.programmaticStreamSerializationAllowed = 1;
        rc.attrs = ra;
        rc.numAttrs = 1;
        e = cudaLaunchKernelEx(&rc, tc_split_reduce_kernel<TOut>, p);
        if (e == cudaSuccess) ++*extra_launches;
    }
    return e;
}

// One operand's 16-bit repack job: dst (rows x ld_dst) from the source's
// rows of K elements; `blocks` is what the job takes of the fused launch.
template <typename TSrc>
PackJob<TSrc> pack_job(const void* src, int64_t ld_src, int64_t rows, int64_t K, void* dst,
                       int64_t ld_dst, int sm_count) {
    PackJob<TSrc> j{};
    j.src = static_cast<const TSrc*>(src);
    j.src_end = j.src + (rows - 1) * ld_src + K;
    j.ld_src = ld_src;
    j.rows = rows;
    j.K = K;
    j.dst = static_cast<uint16_t*>(dst);
    j.ld_dst = ld_dst;
    j.vec_src = (ld_src * static_cast<int64_t>(sizeof(TSrc))) % (8 * sizeof(TSrc)) == 0 &&
                aligned(src, 8 * sizeof(TSrc));
    // one 8-element group per thread where the launch allows (no dependent
    // loads chained through a block-stride loop)
    // a unit is 8 elements of a row per thread (16-bit sources) or 1024
    // elements of a row per warp (int8, see pack_rows_body<int8_t>)
    const int64_t upr = sizeof(TSrc) == 1 ? (ld_dst / 8 + 127) / 128 : ld_dst / 8;
    j.units_per_row = upr;
    const int64_t work = rows * upr;
    const int64_t per_block = sizeof(TSrc) == 1 ? 8 : 256;  // units a block takes at once
    j.blocks = std::max<int64_t>(1, std::min<int64_t>((work + per_block - 1) / per_block,
                                                      static_cast<int64_t>(sm_count) * 256));
    // division by an invariant integer as a multiply and a shift (Granlund and
    // Montgomery): with l = ceil(log2 upr) and m = ceil(2^(31+l) / upr),
    // floor(i / upr) = (i * m) >> (31 + l) for every 0 <= i < 2^31
    j.fast_div = work < (int64_t{1} << 31) ? 1 : 0;
    int l = 0;
    while ((int64_t{1} << l) < upr) ++l;
    j.div_s = 31 + l;
    j.div_m = ((uint64_t{1} << (31 + l)) + static_cast<uint64_t>(upr) - 1) / static_cast<uint64_t>(upr);
    return j;
}

// A transposing int8 job: dst (rows x ld_dst) with dst[r][k] = src[k*ld_src + r]
// for k < K, r < rows; one block per 64 x 128 tile, up to 256 per SM.
PackJob<int8_t> pack_job_transposed(const void* src, int64_t ld_src, int64_t rows, int64_t K,
                                    void* dst, int64_t ld_dst, int sm_count) {
    PackJob<int8_t> j{};
    j.src = static_cast<const int8_t*>(src);
    j.src_end = j.src + (K - 1) * ld_src + rows;
    j.ld_src = ld_src;
    j.rows = rows;
    j.K = K;
    j.dst = static_cast<uint16_t*>(dst);
    j.ld_dst = ld_dst;
    j.vec_src = ld_src % 8 == 0 && aligned(src, 8);
    j.transpose = 1;
    j.tiles_k = (ld_dst + 63) / 64;
    const int64_t tiles = (rows + 127) / 128 * j.tiles_k;
    j.blocks = std::max<int64_t>(1, std::min<int64_t>(tiles, static_cast<int64_t>(sm_count) * 256));
    // tile i -> its 128 rows i / tiles_k through the reciprocal, as for row units
    j.units_per_row = j.tiles_k;
    j.fast_div = tiles < (int64_t{1} << 31) ? 1 : 0;
    int l = 0;
    while ((int64_t{1} << l) < j.tiles_k) ++l;
    j.div_s = 31 + l;
    j.div_m = ((uint64_t{1} << (31 + l)) + static_cast<uint64_t>(j.tiles_k) - 1) /
              static_cast<uint64_t>(j.tiles_k);
    return j;
}

// Launches the repack jobs (either may be absent: blocks = 0) as one grid.
template <typename TSrc>
cudaError_t launch_pack_pair(const PackJob<TSrc>& a, const PackJob<TSrc>& b, cudaStream_t s) {
    const int64_t blocks = a.blocks + b.blocks;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    pack_pair_kernel<TSrc><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a, b);
    return cudaGetLastError();
}

cudaError_t launch_pack_f32(const void* src, int64_t ld_src, bool transposed, int64_t rows,
                            int64_t K, void* dst, int64_t ld_dst, int sm_count, cudaStream_t s) {
    if (transposed) {
        dim3 grid(static_cast<unsigned>((ld_dst + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
        if (grid.y > 65535) return cudaErrorInvalidConfiguration;
        pack_transposed_f32_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(src), ld_src, rows,
                                                        K, static_cast<float*>(dst), ld_dst);
    } else {
        const int64_t work = rows * (ld_dst / 4);
        const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(sm_count) * 16);
        pack_rows_f32_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(
            static_cast<const float*>(src), ld_src, rows, K, static_cast<float*>(dst), ld_dst);
    }
    return cudaGetLastError();
}

}  // namespace

bool tc_supports(const GemmArgs& a) {
    const bool fp = (a.in_dtype == DGA_BF16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_BF16)) ||
                    (a.in_dtype == DGA_F16 && (a.out_dtype == DGA_F32 || a.out_dtype == DGA_F16)) ||
                    (a.in_dtype == DGA_TF32 && a.out_dtype == DGA_F32);
    const bool i8 = a.in_dtype == DGA_I8 && a.out_dtype == DGA_I32;
    if (!fp && !i8) return false;
    if (a.K < 1 || a.M < 1 || a.N < 1) return false;
    // tensor-map extents are 32-bit; tile counts fit comfortably in 32 bits
    if (a.M >= (int64_t(1) << 31) || a.N >= (int64_t(1) << 31) || a.K >= (int64_t(1) << 31)) return false;
    return encode_fn() != nullptr;
}

size_t tc_workspace_size(const GemmArgs& a) {
    PackPlan pl = (a.A && a.B) ? plan_for(a) : plan_for_sizes(a);
    return pl.a_bytes + pl.b_bytes;
}

size_t tc_workspace_wanted(const GemmArgs& a, int sm_count) {
    const size_t need = tc_workspace_size(a);
    // the split last wave (CTA-pair kernel, floating point): at most two
    // rounds of parts on sm_count / 2 clusters; only for more tiles than
    // clusters and K deep enough for two parts
    if (a.in_dtype == DGA_I8 || a.M <= BM || sm_count < 2) return need;
    const int64_t tiles = ((a.M + 255) / 256) * ((a.N + kPairBN - 1) / kPairBN);
    const int64_t kb = (a.K + k_per_stage(a.in_dtype == DGA_TF32 ? kFmtTF32 : kFmtBF16) - 1) /
                       k_per_stage(a.in_dtype == DGA_TF32 ? kFmtTF32 : kFmtBF16);
    if (tiles <= sm_count / 2 || kb < 2 * static_cast<int64_t>(kMinSplitKb)) return need;
    return need + static_cast<size_t>(2 * (sm_count / 2)) * kSplitSlotBytes;
}

cudaError_t tc_launch(const GemmArgs& a, const DeviceInfo& dev, int* launches) {
    const bool i8 = a.in_dtype == DGA_I8;
    const bool tf32 = a.in_dtype == DGA_TF32;
    const bool bf16 = i8 || a.in_dtype == DGA_BF16;
    const uint32_t fmt = tf32 ? kFmtTF32 : (bf16 ? kFmtBF16 : kFmtF16);
    PackPlan pl = plan_for(a);
    if (a.ws_bytes < pl.a_bytes + pl.b_bytes) return cudaErrorInvalidValue;
    const void* A = a.A;
    int64_t lda = a.lda;
    const void* B = a.B;
    int64_t ldb = a.ldb;
    cudaError_t e;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    void* dst_a = ws;
    void* dst_b = ws + pl.a_bytes;
    // TF32 reads K-major operands only: a column-major A or row-major B is
    // transposed into the workspace
    const bool tr_a = a.layout_a == DGA_COL_MAJOR;  // A(i, k) = A[k*lda + i]: to M x K
    const bool tr_b = a.layout_b == DGA_ROW_MAJOR;  // B(k, j) = B[k*ldb + j]: to N x K
    if (tf32) {
        if (pl.pack_a) {
            e = launch_pack_f32(a.A, a.lda, tr_a, a.M, a.K, dst_a, pl.kp, dev.sm_count, a.stream);
            if (e != cudaSuccess) return e;
            ++*launches;
        }
        if (pl.pack_b) {
            e = launch_pack_f32(a.B, a.ldb, tr_b, a.N, a.K, dst_b, pl.kp, dev.sm_count, a.stream);
            if (e != cudaSuccess) return e;
            ++*launches;
        }
    } else if (pl.pack_a || pl.pack_b) {
        // both repacks in one launch; a 16-bit one copies its source row by
        // row (an MN-major operand's rows run along M or N, one per k)
        auto run = [&](auto tag) {
            using T = decltype(tag);
            PackJob<T> ja{}, jb{};
            if (pl.pack_a)
                ja = pl.a_mn ? pack_job<T>(a.A, a.lda, a.K, a.M, dst_a, pl.a_ld, dev.sm_count)
                             : pack_job<T>(a.A, a.lda, a.M, a.K, dst_a, pl.a_ld, dev.sm_count);
            if (pl.pack_b)
                jb = pl.b_mn ? pack_job<T>(a.B, a.ldb, a.K, a.N, dst_b, pl.b_ld, dev.sm_count)
                             : pack_job<T>(a.B, a.ldb, a.N, a.K, dst_b, pl.b_ld, dev.sm_count);
            return launch_pack_pair<T>(ja, jb, a.stream);
        };
        if (i8) {
            // both operands to K-major bf16: column-major A and row-major B
            // are transposed on the way
            PackJob<int8_t> ja = tr_a ? pack_job_transposed(a.A, a.lda, a.M, a.K, dst_a, pl.kp, dev.sm_count)
                                      : pack_job<int8_t>(a.A, a.lda, a.M, a.K, dst_a, pl.kp, dev.sm_count);
            PackJob<int8_t> jb = tr_b ? pack_job_transposed(a.B, a.ldb, a.N, a.K, dst_b, pl.kp, dev.sm_count)
                                      : pack_job<int8_t>(a.B, a.ldb, a.N, a.K, dst_b, pl.kp, dev.sm_count);
            e = launch_pack_pair<int8_t>(ja, jb, a.stream);
        } else {
            e = bf16 ? run(__nv_bfloat16{}) : run(__half{});
        }
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    if (pl.pack_a) {
        A = dst_a;
        lda = pl.a_ld;
    }
    if (pl.pack_b) {
        B = dst_b;
        ldb = pl.b_ld;
    }
    // the GEMM follows a repack: launch it programmatically behind it
    const bool pdl = pl.pack_a || pl.pack_b;
    // Floating point with more than one 128-row tile: the CTA-pair kernel
    // (256 x 256 tiles, each CTA loading half of B).
    // More than one 128-row tile: the CTA-pair kernel (256 x 256 tiles, each
    // CTA loading half of B), INT8 included (its chunked exact accumulation).
    const bool pair = a.M > BM;
    const int BN = pair ? kPairBN : (i8 ? kBnI8 : kBnFloat);
    CUtensorMap ma, mb;
    e = pl.a_mn ? make_mnmajor_map(&ma, A, a.M, a.K, lda, fmt)
                : make_kmajor_map(&ma, A, a.M, a.K, lda, BM, fmt);
    if (e != cudaSuccess) return e;
    e = pl.b_mn ? make_mnmajor_map(&mb, B, a.N, a.K, ldb, fmt)
                : make_kmajor_map(&mb, B, a.N, a.K, ldb, pair ? kPairBN / 2 : BN, fmt);
    if (e != cudaSuccess) return e;

    TcParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.C = a.C;
    p.ldc = a.ldc;
    p.alpha = a.alpha_f;
    p.beta = a.beta_f;
    p.alpha_i = a.alpha_i;
    p.beta_i = a.beta_i;
    p.bias = a.bias;
    p.a_mn = pl.a_mn ? 1u : 0u;
    p.b_mn = pl.b_mn ? 1u : 0u;
    const int tile_m = pair ? 2 * BM : BM;
    p.tiles_m = static_cast<uint32_t>((a.M + tile_m - 1) / tile_m);
    p.tiles_n = static_cast<uint32_t>((a.N + BN - 1) / BN);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.num_kb = static_cast<uint32_t>((a.K + k_per_stage(fmt) - 1) / k_per_stage(fmt));
    p.group_m = raster_group_rows(a.K, p.tiles_m, tile_m);
    p.full_tiles = p.num_tiles;
    p.splits = 1;
    p.num_units = p.num_tiles;

    // workspace past the repacked operands: room for the split last wave
    uint32_t* split_ws = nullptr;
    size_t split_bytes = 0;
    const size_t used = pl.a_bytes + pl.b_bytes;  // multiples of 256 bytes
    if (a.ws != nullptr && a.ws_bytes > used && aligned(static_cast<uint8_t*>(a.ws) + used, 16)) {
        split_ws = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.ws) + used);
        split_bytes = a.ws_bytes - used;
    }
    int extra = 0;  // the split's reduce

    if (i8 && pair) e = launch_pair_kernel<kFmtBF16, true, int32_t>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (i8) e = launch_kernel<kFmtBF16, true, kBnI8, int32_t>(ma, mb, p, dev, a.stream, pdl);
    else if (tf32 && pair) e = launch_pair_kernel<kFmtTF32, false, float>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (tf32) e = launch_kernel<kFmtTF32, false, kBnFloat, float>(ma, mb, p, dev, a.stream, pdl);
    else if (pair && bf16 && a.out_dtype == DGA_F32) e = launch_pair_kernel<kFmtBF16, false, float>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (pair && bf16) e = launch_pair_kernel<kFmtBF16, false, __nv_bfloat16>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (pair && a.out_dtype == DGA_F32) e = launch_pair_kernel<kFmtF16, false, float>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (pair) e = launch_pair_kernel<kFmtF16, false, __half>(ma, mb, p, dev, a.stream, pdl, split_ws, split_bytes, &extra);
    else if (bf16 && a.out_dtype == DGA_F32) e = launch_kernel<kFmtBF16, false, kBnFloat, float>(ma, mb, p, dev, a.stream, pdl);
    else if (bf16) e = launch_kernel<kFmtBF16, false, kBnFloat, __nv_bfloat16>(ma, mb, p, dev, a.stream, pdl);
    else if (a.out_dtype == DGA_F32) e = launch_kernel<kFmtF16, false, kBnFloat, float>(ma, mb, p, dev, a.stream, pdl);
    else e = launch_kernel<kFmtF16, false, kBnFloat, __half>(ma, mb, p, dev, a.stream, pdl);
    if (e == cudaSuccess) *launches += 1 + extra;
    return e;
}

cudaError_t tc_selftest_wait(uint64_t limit_ns, cudaStream_t stream) {
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t tc_status_take(int* status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v != 0) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof zero);
    }
    *status = v;
    return e;
}

}  // namespace dga
