// spmv_csr.cu -- sparse matrix-vector product y <- alpha * A * x + beta * y
// with A in CSR form: the SpMV of "AI Programming: Matrix Product", sections
// "CSR" and "SpMV".  Row i's nonzeros are p in [row_offsets[i],
// row_offsets[i+1]), value values[p] in column column_indices[p]; each is
// multiplied by x[column] and the products of a row are summed.
//
// The page notes that one thread, warp or block per row breaks down when row
// lengths differ a lot (short rows waste lanes, long rows hold up the rest)
// and that implementations split long rows and pack short ones.  This kernel
// does both by construction with a merge-path split: the rows' end offsets
// and the nonzero indices form two sorted lists whose merge has rows + nnz
// items; every warp takes an equal share of that merge, whatever the row
// lengths, and inside a chunk every lane takes 16 consecutive items.
//
//  * Warps are independent workers: no block-wide barrier anywhere, so while
//    one warp waits on its loads the SM runs the others (24 warps per SM:
//    three blocks of eight at up to 85 registers).
//  * Start: a warp finds where its share begins (how many row ends and
//    nonzeros precede it) with a search over row_offsets in which each lane
//    probes one of 32 positions per round: 5 dependent rounds for 4M rows.
//    Its end needs no search: the chunks simply stop at the share's end.
//  * Chunks of 512 merge items (16 per lane: the per-chunk work -- row-end
//    counts, scans, the carry -- is shared by twice the items of 8 per lane,
//    which measured 5.6% faster over the whole call at three blocks per SM;
//    24 per lane at two blocks per SM and 12 per lane at three or four were
//    slower, and 16 per lane at four spilled): in one round trip the warp loads the values
//    and column indices of every nonzero the chunk may hold (coalesced) and
//    the next 32 row ends; a ballot over the row ends' merge positions
//    (row end k sits at k + its end offset within the chunk) counts how many
//    of them fall inside the chunk (more row ends are loaded, 32 at a time,
//    when all do); then it gathers x and keeps the products in shared memory.
//    A chunk's own loads are issued one chunk ahead, as soon as the previous
//    chunk has counted its row ends (which fixes where the next one starts),
//    so they travel while that chunk gathers and sums: a chunk then waits on
//    one round trip, its gathers, instead of two.
//  * Lane ownership: in the usual chunk (at most 32 row ends) lane l holds
//    the nonzeros 16l .. 16l+15 and closes the rows whose last nonzero is
//    among them; it reads its 16 products as four 16-byte vectors (a padding
//    that keeps them on distinct banks) and sums them in registers.  A chunk
//    with more row ends gives each lane 16 consecutive merge items instead, so
//    that no lane closes more than 16 rows.  Either way a shared-memory count
//    of each lane's row ends and a warp prefix sum tell every lane which
//    row ends it closes.  A row
//    that starts and ends inside one lane is written at once; the first row
//    a lane closes may have begun in earlier lanes or chunks, so a warp-wide
//    segmented scan of the lanes' trailing partial sums, seeded with the
//    warp's carry, supplies the missing part.
//  * A row that crosses warp shares is written by the warp that closes it;
//    each earlier warp leaves its partial sum in the workspace (one row index
//    and one float per warp), and a second kernel adds those in warp order.
//    Summation order is fixed: results are reproducible run to run.
//  * alpha and beta follow BLAS: beta == 0 never reads y.  alpha == 0 never
//    reads A or x (a separate scaling kernel runs).
//  * Malformed input never leads to an access outside the arrays: column
//    indices outside [0, cols) and row offsets outside [0, nnz] or out of
//    order are clamped or skipped, and recorded in a status word that
//    dga_sync_status() reports as DGA_ERR_BAD_INDEX.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "dga_internal.h"

namespace dga {

__device__ int g_spmv_status;  // non-zero: the CSR arrays were malformed

namespace {

constexpr int kThreads = 256;
constexpr int kIpt = 16;                     // merge items per lane per chunk
constexpr int kWarpChunk = 32 * kIpt;        // 512 merge items per warp chunk
constexpr int kMaxCtasPerSm = 8;             // 2048 threads per SM; the workspace allows this many

struct SpParams {
    int64_t rows, cols, nnz;
    const int32_t* offs;   // rows + 1 entries
    const int32_t* cidx;   // nnz entries
    const float* vals;     // nnz entries
    const float* x;        // cols entries
    float* y;              // rows entries
    float alpha, beta;
    int64_t items;         // rows + nnz
    int64_t ctas;
    int64_t sms;           // SMs of the device (for the block-to-share mapping)
    int32_t* carry_row;    // workspace: per CTA, the row its last partial sum belongs to
    float* carry_val;      //            and that partial sum
};

__device__ __forceinline__ void flag_bad() { atomicExch(&g_spmv_status, 1); }


// Streamed arrays (values, column indices) are read once: keep them out of L1
// so that L1 holds the x elements the gathers reuse.
__device__ __forceinline__ int32_t ld_stream(const int32_t* q) {
    int32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(q));
    return v;
}
__device__ __forceinline__ float ld_stream(const float* q) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(q));
    return v;
}

// Loads the row ends of rows r + k (k = k0 + lane < k_end; offs_r = the
// row offsets from row r on) into the warp's window as offsets from the
// chunk's first nonzero z, clamped to [0, nz_max]; checks each against the
// offset before it (row offsets must not decrease); returns whether this
// lane's row end falls inside the chunk's n_items.  32-bit throughout: rows
// and nonzeros are below 2^31.
__device__ __forceinline__ bool load_row_ends(const int32_t* offs_r, int nnz, int32_t* endl, int z,
                                              int k0, int k_end, int nz_max, int n_items) {
    const int lane = threadIdx.x & 31;
    const int k = k0 + lane;
    int raw = 0;
    if (k < k_end) raw = offs_r[k + 1];
    // the offset before: the previous lane's, or for lane 0 the row start
    int before = __shfl_up_sync(0xffffffffu, raw, 1);
    if (lane == 0 && k < k_end) before = offs_r[k];
    if (k < k_end && raw < before) flag_bad();
    if (k >= k_end) return false;
    if (raw < 0 || raw > nnz) flag_bad();
    const int e = min(min(max(raw, 0), nnz) - z, nz_max);
    endl[k] = e < 0 ? 0 : e;
    return k + endl[k] < n_items;
}

// The same in two halves, so that a chunk's first window of row ends can be
// loaded while the previous chunk is still being processed: the loads
// (this lane's row end and, for lane 0, the offset before the window) ...
__device__ __forceinline__ void row_ends_issue(const int32_t* offs_r, int k_end, int& raw,
                                               int& before0) {
    const int lane = threadIdx.x & 31;
    raw = 0;
    before0 = 0;
    if (lane < k_end) {
        raw = offs_r[lane + 1];
        if (lane == 0) before0 = offs_r[0];
    }
}

// ... and the rest, once the chunk's first nonzero z is known.
__device__ __forceinline__ bool row_ends_consume(int raw, int before0, int nnz, int32_t* endl, int z,
                                                 int k_end, int nz_max, int n_items) {
    const int lane = threadIdx.x & 31;
    int before = __shfl_up_sync(0xffffffffu, raw, 1);
    if (lane == 0) before = before0;
    if (lane < k_end && raw < before) flag_bad();
    if (lane >= k_end) return false;
    if (raw < 0 || raw > nnz) flag_bad();
    const int e = min(min(max(raw, 0), nnz) - z, nz_max);
    endl[lane] = e < 0 ? 0 : e;
    return lane + endl[lane] < n_items;
}

// Row end i (i < rows) as a position in the nonzero list, clamped to [0, nnz].
__device__ __forceinline__ int64_t row_end(const SpParams& p, int64_t i) {
    int64_t v = p.offs[i + 1];
    if (v < 0 || v > p.nnz) {
        flag_bad();
        v = v < 0 ? 0 : p.nnz;
    }
    return v;
}

// Number of row ends among the first d merge items: the smallest i in
// [max(0, d - nnz), min(d, rows)] such that row end i is not taken, where row
// end i is taken before nonzero j when end(i) <= j, and the j competing with
// row end i on diagonal d is d - 1 - i.  Taken positions form a prefix.  The
// whole warp searches: each lane probes one of 32 evenly spread positions per
// round (every round narrows the interval 32-fold), and every lane returns
// the same answer.
__device__ int64_t warp_merge_search(const SpParams& p, int64_t d) {
    const int lane = threadIdx.x & 31;
    int64_t lo = d > p.nnz ? d - p.nnz : 0;
    int64_t hi = d < p.rows ? d : p.rows;
    while (lo < hi) {  // at most 7 rounds for 2^31 rows
        const int64_t q = lo + (hi - lo) * lane / 32;  // q_0 = lo, nondecreasing in lane
        const bool taken = row_end(p, q) <= d - 1 - q;
        const int c = __popc(__ballot_sync(0xffffffffu, taken));
        // probes 0 .. c-1 are taken: the answer lies in [q_{c-1} + 1, q_c]
        const int64_t nlo = c > 0 ? lo + (hi - lo) * (c - 1) / 32 + 1 : lo;
        const int64_t nhi = c < 32 ? lo + (hi - lo) * c / 32 : hi;
        lo = nlo;
        hi = nhi;
    }
    return lo;
}

// Shared-memory index of product k: one padding slot per 32 keeps the
// lanes' contiguous runs (8 apart) on different banks.
__device__ __forceinline__ int pad(int k) { return k + (k >> 5); }

// Per-warp shared memory.
struct WarpSmem {
    int32_t endl[kWarpChunk];              // chunk rows' end offsets, relative to the chunk's first nonzero
    // products of the chunk's nonzeros, padded (pad(k), or padv(k) in chunks
    // read by nonzero ownership: see the kernel)
    __align__(16) float prod[kWarpChunk + kWarpChunk / 8];
    int owned[32];                         // row ends among each lane's items
};

// Shared-memory index of product k when lane l reads its products
// kIpt*l .. kIpt*l + kIpt - 1 as 16-byte vectors: 4 floats of padding per 32
// put the 8 lanes of each quarter-warp phase on 8 different 4-bank groups
// (lane l's run starts at 16l + 4 * (l / 2): bank group 4l + l/2 mod 8).
__device__ __forceinline__ int padv(int k) { return k + ((k >> 5) << 2); }

__global__ void __launch_bounds__(kThreads, 3) spmv_merge_kernel(SpParams p) {
    __shared__ WarpSmem s_all[kThreads / 32];
    const int lane = threadIdx.x & 31;
    WarpSmem& sm = s_all[threadIdx.x >> 5];
    const int64_t warps = p.ctas * (kThreads / 32);
    // Blocks b, b + sms, b + 2 sms, ... usually share an SM (one wave, placed
    // round-robin): give them adjacent shares of the merge, so that the x
    // elements their gathers touch overlap in that SM's L1.  Any mapping is
    // correct (a permutation of the shares); this one is only faster.
    // (b = q * sms + s maps to s * per_sm + q: a bijection when sms divides ctas)
    const int64_t b = blockIdx.x;
    const int64_t per_sm = p.ctas / p.sms;
    const int64_t logical = p.ctas % p.sms == 0 ? (b % p.sms) * per_sm + b / p.sms : b;
    const int64_t w = logical * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t d_begin = w * p.items / warps;
    const int64_t r0 = warp_merge_search(p, d_begin);
    if (w == 0 && lane == 0 && p.rows > 0 &&
        (p.offs[0] != 0 || static_cast<int64_t>(p.offs[p.rows]) != p.nnz))
        flag_bad();
    // rows and nonzeros are below 2^31 (the entry point checks), and a share
    // holds at most items / 8 < 2^29 merge items: 32-bit counters from here
    const int rows = static_cast<int>(p.rows), nnz = static_cast<int>(p.nnz);
    int r = static_cast<int>(r0), z = static_cast<int>(d_begin - r0);
    int left = static_cast<int>((w + 1) * p.items / warps - d_begin);  // merge items still to do
    float carry = 0.0f;  // partial sum of row r carried from earlier chunks of this warp

    // A chunk's loads: the values and column indices of every nonzero it may
    // hold (those past its split are read again, from L1/L2, by the next
    // chunk) and its first 32 row ends.  They are issued one chunk ahead --
    // while the previous chunk gathers x and sums -- so that a chunk waits on
    // one round trip (its gathers) instead of two.
    // (entries past a chunk's nonzeros keep stale values: only the first c_nz
    // are ever read, so they are set once here rather than every chunk)
    int32_t col[kIpt] = {};
    float val[kIpt] = {};
    int raw0 = 0, before0 = 0;
    auto issue = [&](int zz, int rr, int nzm, int win0) {
        // one base address per array, the 32-element steps as constant offsets
        const int32_t* cb = p.cidx + zz + lane;
        const float* vb = p.vals + zz + lane;
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            if (u * 32 + lane < nzm) {
                col[u] = ld_stream(cb + u * 32);
                val[u] = ld_stream(vb + u * 32);
            }
        }
        row_ends_issue(p.offs + rr, win0, raw0, before0);
    };
    int n_items = min(kWarpChunk, left);
    int rows_max = min(n_items, rows - r);  // row ends the chunk may hold
    int nz_max = min(n_items, nnz - z);     // nonzeros the chunk may hold
    if (left > 0) issue(z, r, nz_max, min(32, rows_max));

    while (left > 0) {
        const int32_t* offs_r = p.offs + r;
        float* y_r = p.y + r;
        // row end k sits at merge position k + (its end - z) of the chunk;
        // those inside the chunk are a prefix of the rows
        int win = min(32, rows_max);
        int c_rows = __popc(__ballot_sync(
            0xffffffffu, row_ends_consume(raw0, before0, nnz, sm.endl, z, win, nz_max, n_items)));
        while (c_rows == win && win < rows_max) {  // every row of the window closes: widen it
            const int k0 = win;
            win = min(win + 32, rows_max);
            c_rows += __popc(__ballot_sync(
                0xffffffffu, load_row_ends(offs_r, nnz, sm.endl, z, k0, win, nz_max, n_items)));
        }
        int c_nz = n_items - c_rows;
        if (c_nz > nz_max) {  // only for malformed offsets: keep every index in range
            flag_bad();
            c_nz = nz_max;
        }
        // Which lane closes which row (warp-uniform choice).  A chunk with at
        // most 32 row ends (the usual case) gives lane l the nonzeros
        // [16l, 16l + 16) and each row end to the lane holding the row's last
        // nonzero (lane 0 for a row with none in the chunk); the lane reads
        // its 16 products as four 16-byte vectors and sums them in registers.
        // A chunk with more row ends (mostly empty rows) gives lane l the
        // merge items [16l, 16l + 16) instead, row ends included, so that no
        // lane closes more than 16 rows.
        const bool by_nz = c_rows <= 32;
        // gather x (the loads first, all in flight together)
        float xv[kIpt];
        const uint32_t ucols = static_cast<uint32_t>(p.cols);  // cols < 2^31
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            xv[u] = 0.0f;
            if (u * 32 + lane < c_nz) {
                // one unsigned compare: a negative index is a large unsigned one
                if (static_cast<uint32_t>(col[u]) < ucols) xv[u] = __ldg(p.x + col[u]);
                else flag_bad();
            }
        }
        // this chunk's products, then the next chunk's loads (in flight while
        // this chunk is summed and written)
        // zero past the chunk's nonzeros, so that a lane reading all its
        // products by vector finds zeros there (a select, not val * 0: an
        // infinite value of the next chunk would make a NaN).  Product
        // u * 32 + lane sits at padv = lane + 36u or pad = lane + 33u: one
        // base address and constant offsets per ownership mode.
        if (by_nz) {
            float* pb = sm.prod + lane;
#pragma unroll
            for (int u = 0; u < kIpt; ++u) pb[36 * u] = u * 32 + lane < c_nz ? val[u] * xv[u] : 0.0f;
        } else {
            float* pb = sm.prod + lane;
#pragma unroll
            for (int u = 0; u < kIpt; ++u) pb[33 * u] = u * 32 + lane < c_nz ? val[u] * xv[u] : 0.0f;
        }
        const int chunk_items = n_items, chunk_nz = c_nz;
        const int r_next = r + c_rows, z_next = z + c_nz, left_next = left - (c_rows + c_nz);
        if (left_next > 0) {
            n_items = min(kWarpChunk, left_next);
            rows_max = min(n_items, rows - r_next);
            nz_max = min(n_items, nnz - z_next);
            issue(z_next, r_next, nz_max, min(32, rows_max));
        }
        sm.owned[lane] = 0;
        __syncwarp();
        for (int k = lane; k < c_rows; k += 32) {
            const int e = sm.endl[k];
            const int owner = by_nz ? (e > 0 ? (e - 1) / kIpt : 0) : min(k + e, chunk_items - 1) / kIpt;
            atomicAdd(&sm.owned[owner], 1);
        }
        __syncwarp();

        // --- this lane's row ends rs .. re-1 (from the counts), and the
        // nonzeros before, between and after them
        const int owned = sm.owned[lane];
        int incl = owned;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int up = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += up;
        }
        const int rs = incl - owned;
        const int re = min(incl, c_rows);
        float run = 0.0f, head = 0.0f;
        // closes row end k with the running sum: the lane's first row end
        // (which may have begun in earlier lanes) waits for the scan below
        auto close_row = [&](int k) {
            if (k == rs) {
                head = run;
            } else {
                float* dst = y_r + k;  // the whole row lies in this lane's items
                const float old = p.beta != 0.0f ? *dst : 0.0f;
                *dst = fmaf(p.beta, old, p.alpha * run);
            }
            run = 0.0f;
        };
        if (by_nz) {
            const int base = lane * kIpt;
            float pv[kIpt];
#pragma unroll
            for (int q = 0; q < kIpt / 4; ++q) {
                const float4 v4 = *reinterpret_cast<const float4*>(&sm.prod[padv(base) + 4 * q]);
                pv[4 * q] = v4.x;
                pv[4 * q + 1] = v4.y;
                pv[4 * q + 2] = v4.z;
                pv[4 * q + 3] = v4.w;
            }
            // row end k (rs <= k < re) closes before product endl[k] - base,
            // a position in 0 .. kIpt
            if (!__any_sync(0xffffffffu, re - rs > 2)) {
                // No lane closes more than two rows (the usual chunk): one
                // straight pass over the products with the two cut positions
                // as predicated resets, in the same order of additions as the
                // general loop below, so the sums are the same bits -- without
                // its branches, which the warp takes at almost every step
                // because some lane closes a row there.
                const int n_ends = re - rs;
                const int a1 = n_ends >= 1 ? sm.endl[rs] - base : -1;
                const int a2 = n_ends >= 2 ? sm.endl[rs + 1] - base : -1;
                float mid = 0.0f;
#pragma unroll
                for (int t = 0; t <= kIpt; ++t) {
                    if (a1 == t) {
                        head = run;
                        run = 0.0f;
                    }
                    if (a2 == t) {
                        mid = run;
                        run = 0.0f;
                    }
                    if (t < kIpt) run += pv[t];
                }
                if (n_ends >= 2) {
                    float* dst = y_r + rs + 1;  // the whole row lies in this lane's items
                    const float old = p.beta != 0.0f ? *dst : 0.0f;
                    *dst = fmaf(p.beta, old, p.alpha * mid);
                }
            } else {
                int k = rs;
                int at = k < re ? sm.endl[k] - base : kIpt + 1;
#pragma unroll
                for (int t = 0; t < kIpt; ++t) {
                    while (at == t) {
                        close_row(k);
                        ++k;
                        at = k < re ? sm.endl[k] - base : kIpt + 1;
                    }
                    run += pv[t];
                }
                while (at == kIpt) {
                    close_row(k);
                    ++k;
                    at = k < re ? sm.endl[k] - base : kIpt + 1;
                }
            }
        } else {
            const int items_here = max(0, min(kIpt, chunk_items - lane * kIpt));
            int nz = min(max(lane * kIpt - rs, 0), chunk_nz);
            const int nz_end = min(max(nz + items_here - owned, nz), chunk_nz);
            for (int k = rs; k < re; ++k) {
                const int e = min(max(sm.endl[k], nz), nz_end);
                for (; nz < e; ++nz) run += sm.prod[pad(nz)];
                close_row(k);
            }
            for (; nz < nz_end; ++nz) run += sm.prod[pad(nz)];
        }

        // --- segmented scan of (has_end, tail) over the lanes, the warp's
        // carry first: combine(a, b) = (a.f | b.f, b.f ? b.v : a.v + b.v)
        const int has_end = re > rs ? 1 : 0;
        int f = has_end;
        float v = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float v_up = __shfl_up_sync(0xffffffffu, v, off);
            const int f_up = __shfl_up_sync(0xffffffffu, f, off);
            if (lane >= off) {
                if (!f) v += v_up;
                f |= f_up;
            }
        }
        // exclusive prefix of this lane: the carry combined with lanes before it
        const float lane_v = __shfl_up_sync(0xffffffffu, v, 1);
        const int lane_f = __shfl_up_sync(0xffffffffu, f, 1);
        const float carry_in = lane == 0 ? carry : (lane_f ? lane_v : carry + lane_v);
        if (has_end) {
            float* dst = y_r + rs;
            const float old = p.beta != 0.0f ? *dst : 0.0f;
            *dst = fmaf(p.beta, old, p.alpha * (carry_in + head));
        }
        // the chunk's outgoing carry: the scan total
        const float tot_v = __shfl_sync(0xffffffffu, v, 31);
        const int tot_f = __shfl_sync(0xffffffffu, f, 31);
        carry = tot_f ? tot_v : carry + tot_v;
        r = r_next;
        z = z_next;
        left = left_next;
        __syncwarp();  // the warp's shared arrays are reused by the next chunk
    }
    if (lane == 0) {
        // row r has not closed in this warp: its partial sum goes to the next one
        p.carry_row[w] = r;
        p.carry_val[w] = carry;
    }
}

// Adds each warp's trailing partial sum (times alpha) to its row; runs of
// warps that end inside the same row are summed in warp order by the run's
// first thread.
__global__ void spmv_fixup_kernel(SpParams p) {
    const int64_t warps = p.ctas * (kThreads / 32);
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < warps;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t row = p.carry_row[c];
        if (c > 0 && p.carry_row[c - 1] == row) continue;  // not the first of its run
        if (row < 0 || row >= p.rows) continue;            // past the last row: nothing to add
        float s = 0.0f;
        for (int64_t k = c; k < warps && p.carry_row[k] == row; ++k) s += p.carry_val[k];
        p.y[row] += p.alpha * s;
    }
}

// alpha == 0 (or no nonzeros to read): y <- beta * y, y <- 0 when beta == 0.
__global__ void spmv_scale_kernel(float* y, int64_t rows, float beta) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        y[i] = beta != 0.0f ? beta * y[i] : 0.0f;
}

// CTAs of the merge kernel: one wave of as many as fit on the device (queried
// once per device), no more than there are chunks.  ctas_per_sm <= 0: the
// upper bound the workspace is sized for.
int64_t spmv_ctas(int64_t items, int sm_count, int ctas_per_sm) {
    const int per_sm = ctas_per_sm > 0 ? std::min(ctas_per_sm, kMaxCtasPerSm) : kMaxCtasPerSm;
    const int64_t full = static_cast<int64_t>(sm_count > 0 ? sm_count : 152) * per_sm;
    const int64_t needed = (items + kThreads * kIpt - 1) / (kThreads * kIpt);
    return std::max<int64_t>(1, std::min(full, needed));
}

int merge_ctas_per_sm(const DeviceInfo& dev) {
    static int cached[64] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    const bool cacheable = dev.ordinal >= 0 && dev.ordinal < 64;
    if (cacheable && cached[dev.ordinal] > 0) return cached[dev.ordinal];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, spmv_merge_kernel, kThreads, 0) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        n = 4;
    }
    if (cacheable) cached[dev.ordinal] = n;
    return n;
}

}  // namespace

size_t spmv_workspace_size(int64_t rows, int64_t nnz, int sm_count) {
    const int64_t warps = spmv_ctas(rows + nnz, sm_count, 0) * (kThreads / 32);
    return static_cast<size_t>(warps) * (sizeof(int32_t) + sizeof(float)) + 256;
}

cudaError_t spmv_launch(int64_t rows, int64_t cols, int64_t nnz, const int32_t* row_offsets,
                        const int32_t* column_indices, const float* values, float alpha,
                        const float* x, float beta, float* y, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t stream, int* launches) {
    if (alpha == 0.0f || nnz == 0) {
        // no products to form: y <- beta * y (alpha * A x is zero)
        const int64_t blocks = std::min<int64_t>((rows + 255) / 256, static_cast<int64_t>(dev.sm_count) * 8);
        spmv_scale_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(y, rows, beta);
        ++*launches;
        return cudaGetLastError();
    }
    SpParams p{};
    p.rows = rows;
    p.cols = cols;
    p.nnz = nnz;
    p.offs = row_offsets;
    p.cidx = column_indices;
    p.vals = values;
    p.x = x;
    p.y = y;
    p.alpha = alpha;
    p.beta = beta;
    p.items = rows + nnz;
    p.ctas = spmv_ctas(p.items, dev.sm_count, merge_ctas_per_sm(dev));
    p.sms = std::max(1, dev.sm_count);
    if (ws_bytes < spmv_workspace_size(rows, nnz, dev.sm_count)) return cudaErrorInvalidValue;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.carry_row = reinterpret_cast<int32_t*>(w);
    p.carry_val = reinterpret_cast<float*>(w + ((p.ctas * (kThreads / 32) * sizeof(int32_t) + 127) / 128) * 128);
    spmv_merge_kernel<<<static_cast<unsigned>(p.ctas), kThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    spmv_fixup_kernel<<<static_cast<unsigned>((p.ctas * (kThreads / 32) + 255) / 256), 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e == cudaSuccess) *launches += 2;
    return e;
}

cudaError_t spmv_status_take(int* status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_spmv_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v != 0) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_spmv_status, &zero, sizeof zero);
    }
    *status = v;
    return e;
}

}  // namespace dga
