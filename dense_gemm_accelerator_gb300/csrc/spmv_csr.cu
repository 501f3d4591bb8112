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
// items; every CTA takes an equal share of that merge, whatever the row
// lengths, and inside it every thread takes 8 consecutive items.
//
//  * CTA range: the start of a CTA's share (how many row ends and nonzeros
//    precede it) comes from a cooperative search over row_offsets: each of
//    128 threads probes one position per round, so 4 dependent rounds cover
//    2^28 rows.  The two ends of the range are searched at once.
//  * Chunks of 2048 merge items: in one round trip the CTA loads the chunk's
//    first 256 row ends and the values and column indices of every nonzero
//    the chunk may hold (coalesced), then gathers x for them and keeps the
//    products in shared memory; one barrier count over the row ends' merge
//    positions gives how many of the items are row ends (the row-end window
//    grows in steps of 256 when a chunk holds more rows).  HBM traffic is about one pass over values,
//    column indices and row offsets; x is gathered through L1/L2.
//  * Each thread owns 8 consecutive merge items.  Row end k sits at merge
//    position k + (its end offset - the chunk's first nonzero), so one
//    shared-memory count per row end tells every thread how many row ends it
//    owns, and a block-wide prefix sum where they start; a thread then sums
//    the products between its row ends (a tight loop over shared memory,
//    padded so that the threads' runs fall on different banks).  A row that starts
//    and ends inside one thread is written at once; the first row a thread
//    closes may have begun in earlier threads, so a block-wide segmented scan
//    of the threads' trailing partial sums supplies the missing part.  The
//    chunk's last partial row carries into the next chunk.
//  * A row that crosses CTA ranges is written by the CTA that closes it; each
//    earlier CTA leaves its partial sum in the workspace (one row index and
//    one float per CTA), and a second kernel adds those in CTA order.
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
constexpr int kIpt = 8;                      // merge items per thread per chunk
constexpr int kChunk = kThreads * kIpt;      // 2048 merge items per chunk
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
    int32_t* carry_row;    // workspace: per CTA, the row its last partial sum belongs to
    float* carry_val;      //            and that partial sum
};

__device__ __forceinline__ void flag_bad() { atomicExch(&g_spmv_status, 1); }

__device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

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
// row end i on diagonal d is d - 1 - i.  Taken positions form a prefix.
// `half` (0 or 1) picks which half of the CTA's threads searches this d; each
// half probes 128 positions per round, so every round narrows the interval
// 128-fold.  Every thread of the CTA calls this (it holds barriers).
__device__ int64_t merge_search(const SpParams& p, int64_t d, int half, int64_t* s_bounds,
                                int* s_cnt) {
    const int t = threadIdx.x & 127;
    int64_t* b = s_bounds + 2 * half;
    if (t == 0) {
        b[0] = d > p.nnz ? d - p.nnz : 0;
        b[1] = d < p.rows ? d : p.rows;
    }
    __syncthreads();
    for (int round = 0; round < 6; ++round) {  // 128^5 > 2^31 rows
        const int64_t lo = b[0], hi = b[1];
        bool taken = false;
        if (lo < hi) {
            const int64_t q = lo + (hi - lo) * t / 128;  // q_0 = lo, nondecreasing in t
            taken = row_end(p, q) <= d - 1 - q;
        }
        const unsigned m = __ballot_sync(0xffffffffu, taken);
        if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = __popc(m);
        __syncthreads();
        if (t == 0 && lo < hi) {
            int c = 0;
            for (int k = 0; k < 4; ++k) c += s_cnt[half * 4 + k];
            // probes 0 .. c-1 are taken: the answer lies in [q_{c-1} + 1, q_c]
            b[0] = c > 0 ? lo + (hi - lo) * (c - 1) / 128 + 1 : lo;
            b[1] = c < 128 ? lo + (hi - lo) * c / 128 : hi;
        }
        __syncthreads();
    }
    return b[0];
}

// Shared-memory index of product k: one padding slot per 32 keeps the
// threads' contiguous runs (8 apart) on different banks.
__device__ __forceinline__ int pad(int k) { return k + (k >> 5); }

// Exclusive prefix sum of v over the CTA's threads (warp shuffles, then the
// warp totals through shared memory); *total receives the sum of all.
__device__ __forceinline__ int block_exclusive_sum(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += up;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) before += s_warp[w];
        all += s_warp[w];
    }
    *total = all;
    return before + incl - v;
}

__global__ void __launch_bounds__(kThreads, 6) spmv_merge_kernel(SpParams p) {
    __shared__ int64_t s_bounds[4];
    __shared__ int s_cnt[kThreads / 32];
    __shared__ int64_t s_range[4];           // r0, z0, r1, z1 of this CTA
    __shared__ int32_t s_endl[kChunk];       // chunk rows' end offsets, relative to the chunk's first nonzero
    __shared__ float s_prod[kChunk + kChunk / 32];  // products of the chunk's nonzeros (padded)
    __shared__ int s_owned[kThreads];        // row ends among each thread's 8 items
    __shared__ int s_warp_i[kThreads / 32];
    __shared__ float s_warp_v[kThreads / 32];
    __shared__ int s_warp_f[kThreads / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t d0 = static_cast<int64_t>(blockIdx.x) * p.items / p.ctas;
    const int64_t d1 = (static_cast<int64_t>(blockIdx.x) + 1) * p.items / p.ctas;

    // --- the CTA's range: threads 0-127 search d0, threads 128-255 search d1
    {
        const int half = tid >> 7;
        const int64_t r = merge_search(p, half ? d1 : d0, half, s_bounds, s_cnt);
        if ((tid & 127) == 0) {
            s_range[2 * half] = r;
            s_range[2 * half + 1] = (half ? d1 : d0) - r;
        }
        __syncthreads();
    }
    int64_t r = s_range[0], z = s_range[1];
    const int64_t r1 = s_range[2], z1 = s_range[3];
    if (blockIdx.x == 0 && tid == 0 && p.rows > 0 &&
        (p.offs[0] != 0 || static_cast<int64_t>(p.offs[p.rows]) != p.nnz))
        flag_bad();
    float carry = 0.0f;  // partial sum of row r carried from earlier chunks of this CTA

    while (r + z < d1) {
        const int n_items = static_cast<int>(lmin(kChunk, d1 - (r + z)));
        const int rows_max = static_cast<int>(lmin(n_items, r1 - r));  // row ends the chunk may hold
        const int nz_max = static_cast<int>(lmin(n_items, z1 - z));     // nonzeros it may hold
        // One round trip for everything the chunk may need: the first 256 row
        // ends (rows average far fewer items than that; more are loaded below
        // when not), and values and column indices of every nonzero it may
        // hold (those past its split are read again, from L2, by the next chunk).
        int32_t col[kIpt];
        float val[kIpt];
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            const int k = u * kThreads + tid;
            col[u] = -1;
            val[u] = 0.0f;
            if (k < nz_max) {
                col[u] = __ldg(p.cidx + z + k);
                val[u] = __ldg(p.vals + z + k);
            }
        }
        // row end k sits at merge position k + (its end - z) of the chunk
        int win = min(kThreads, rows_max);
        bool in_chunk = false;
        if (tid < win) {
            const int e = static_cast<int>(lmin(row_end(p, r + tid) - z, nz_max));
            s_endl[tid] = max(e, 0);
            in_chunk = tid + max(e, 0) < n_items;
        }
        s_owned[tid] = 0;
#pragma unroll
        for (int u = 0; u < kIpt; ++u) {
            const int k = u * kThreads + tid;
            if (k < nz_max) {
                float xv = 0.0f;
                if (col[u] >= 0 && col[u] < p.cols) xv = __ldg(p.x + col[u]);
                else flag_bad();
                s_prod[pad(k)] = val[u] * xv;
            }
        }
        // rows whose end falls inside the chunk: a prefix of the window
        int c_rows = __syncthreads_count(in_chunk);
        while (c_rows == win && win < rows_max) {  // every row of the window closes: widen it
            const int k = win + tid;
            in_chunk = false;
            if (k < rows_max) {
                const int e = static_cast<int>(lmin(row_end(p, r + k) - z, nz_max));
                s_endl[k] = max(e, 0);
                in_chunk = k + max(e, 0) < n_items;
            }
            win = min(win + kThreads, rows_max);
            c_rows += __syncthreads_count(in_chunk);
        }
        int c_nz = n_items - c_rows;
        if (c_nz > nz_max) {  // only for malformed offsets: keep every index in range
            flag_bad();
            c_nz = nz_max;
        }
        for (int k = tid; k < c_rows; k += kThreads) {
            if (k > 0 && s_endl[k] < s_endl[k - 1]) flag_bad();  // row offsets out of order
            const int pos = min(k + s_endl[k], n_items - 1);
            atomicAdd(&s_owned[pos >> 3], 1);  // the thread whose 8 items hold this row end
        }
        __syncthreads();

        // --- this thread's items [tid*8, tid*8 + 8): row ends rs .. re-1, and
        // the nonzeros before, between and after them
        const int owned = s_owned[tid];
        int all_owned;
        const int rs = block_exclusive_sum(owned, s_warp_i, &all_owned);
        const int re = min(rs + owned, c_rows);
        const int items_here = max(0, min(kIpt, n_items - tid * kIpt));
        int nz = min(max(tid * kIpt - rs, 0), c_nz);
        const int nz_end = min(max(nz + items_here - owned, nz), c_nz);
        float run = 0.0f, head = 0.0f;
        for (int k = rs; k < re; ++k) {
            const int e = min(max(s_endl[k], nz), nz_end);
            for (; nz < e; ++nz) run += s_prod[pad(nz)];
            if (k == rs) {
                head = run;  // closes a row that may have begun in earlier threads
            } else {
                float* dst = p.y + (r + k);  // the whole row lies in this thread's items
                const float old = p.beta != 0.0f ? *dst : 0.0f;
                *dst = fmaf(p.beta, old, p.alpha * run);
            }
            run = 0.0f;
        }
        for (; nz < nz_end; ++nz) run += s_prod[pad(nz)];

        // --- segmented exclusive scan of (has_end, tail) over the threads:
        // combine(a, b) = (a.f | b.f, b.f ? b.v : a.v + b.v)
        int f = re > rs ? 1 : 0;
        const int has_end = f;
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
        if (lane == 31) {
            s_warp_v[warp] = v;
            s_warp_f[warp] = f;
        }
        __syncthreads();
        // exclusive prefix: the chunk carry and earlier warps, then earlier lanes
        float pre_v = carry;
        for (int w = 0; w < warp; ++w) {
            if (s_warp_f[w]) pre_v = s_warp_v[w];
            else pre_v += s_warp_v[w];
        }
        const float lane_v = __shfl_up_sync(0xffffffffu, v, 1);
        const int lane_f = __shfl_up_sync(0xffffffffu, f, 1);
        float carry_in = pre_v;
        if (lane > 0) carry_in = lane_f ? lane_v : pre_v + lane_v;
        if (has_end) {
            float* dst = p.y + (r + rs);
            const float old = p.beta != 0.0f ? *dst : 0.0f;
            *dst = fmaf(p.beta, old, p.alpha * (carry_in + head));
        }
        // the chunk's outgoing carry: the scan total
        float total = carry;
        for (int w = 0; w < kThreads / 32; ++w) {
            if (s_warp_f[w]) total = s_warp_v[w];
            else total += s_warp_v[w];
        }
        carry = total;
        r += c_rows;
        z += c_nz;
        __syncthreads();  // shared arrays are reused by the next chunk
    }
    if (tid == 0) {
        // row r has not closed in this CTA: its partial sum goes to the next one
        p.carry_row[blockIdx.x] = static_cast<int32_t>(lmin(r, 0x7fffffff));
        p.carry_val[blockIdx.x] = carry;
    }
}

// Adds each CTA's trailing partial sum (times alpha) to its row; runs of CTAs
// that end inside the same row are summed in CTA order by the run's first
// thread.
__global__ void spmv_fixup_kernel(SpParams p) {
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < p.ctas;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t row = p.carry_row[c];
        if (c > 0 && p.carry_row[c - 1] == row) continue;  // not the first of its run
        if (row < 0 || row >= p.rows) continue;            // past the last row: nothing to add
        float s = 0.0f;
        for (int64_t k = c; k < p.ctas && p.carry_row[k] == row; ++k) s += p.carry_val[k];
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
    const int64_t needed = (items + kChunk - 1) / kChunk;
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
    const int64_t ctas = spmv_ctas(rows + nnz, sm_count, 0);
    return static_cast<size_t>(ctas) * (sizeof(int32_t) + sizeof(float)) + 256;
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
    if (ws_bytes < spmv_workspace_size(rows, nnz, dev.sm_count)) return cudaErrorInvalidValue;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.carry_row = reinterpret_cast<int32_t*>(w);
    p.carry_val = reinterpret_cast<float*>(w + ((p.ctas * sizeof(int32_t) + 127) / 128) * 128);
    spmv_merge_kernel<<<static_cast<unsigned>(p.ctas), kThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    spmv_fixup_kernel<<<static_cast<unsigned>((p.ctas + 255) / 256), 256, 0, stream>>>(p);
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
