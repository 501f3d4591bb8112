// sum_rows.cu -- column sums out[j] = sum over i of G(i, j), in fp32: the
// bias gradient of the fully-connected layer ("AI Programming: Matrix
// Product", section "Fully-connected layer": the output gradient summed over
// the batch).  Bandwidth-bound: every element of G is read once.
//
// Layout of the work:
//   * a CTA owns 32 x VEC consecutive columns (VEC = 16 bytes of elements:
//     8 for bf16/fp16, 4 for fp32); each lane loads 16 bytes, so one warp
//     load is a contiguous 512-byte row segment;
//   * the 8 CTAs of a thread-block cluster split the rows into 8 contiguous
//     slices; inside a CTA, warp w of 16 takes rows w, w + 16, ... of its
//     slice, eight rows in flight per warp (8 warps per CTA measured 58% of
//     DRAM peak on an 8192 x 8192 bf16 gradient, latency-bound);
//   * partial sums are combined in a fixed order -- the 16 warps of a CTA
//     through shared memory, then the 8 CTAs of the cluster by rank 0
//     reading the others' shared memory (distributed shared memory) -- so
//     the result does not depend on timing, and no workspace or atomics are
//     needed.
// Columns past the last whole 16-byte group, or a G whose rows are not
// 16-byte aligned, take element-wise loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dga_internal.h"
#include "ptx.cuh"

namespace dga {
namespace {

constexpr int kWarps = 16;  // 512 threads: enough 16-byte loads in flight to cover HBM latency
constexpr int kCluster = 8;  // CTAs per cluster (portable size)
constexpr int kUnroll = 8;   // rows in flight per warp

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;
    __device__ static void add(const uint4& v, float* acc) {
        acc[0] += __uint_as_float(v.x);
        acc[1] += __uint_as_float(v.y);
        acc[2] += __uint_as_float(v.z);
        acc[3] += __uint_as_float(v.w);
    }
    __device__ static float one(const float* p) { return *p; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static void add(const uint4& v, float* acc) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // a bf16 is the top half of an fp32
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};
template <> struct Elem<__half> {
    static constexpr int kVec = 8;
    __device__ static void add(const uint4& v, float* acc) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            const float2 f = __half22float2(h);
            acc[2 * i] += f.x;
            acc[2 * i + 1] += f.y;
        }
    }
    __device__ static float one(const __half* p) { return __half2float(*p); }
};

template <typename T>
__global__ void __cluster_dims__(1, kCluster, 1) __launch_bounds__(kWarps * 32)
    sum_rows_kernel(const T* __restrict__ G, int64_t rows, int64_t cols, int64_t ldg,
                    float* __restrict__ out, int vec_ok) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int kCols = 32 * VEC;
    __shared__ float part[kWarps][kCols];
    __shared__ float total[kCols];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kCols + lane * VEC;
    const int64_t per = (rows + kCluster - 1) / kCluster;
    const int64_t r_begin = min(rows, static_cast<int64_t>(rank) * per);
    const int64_t r_end = min(rows, r_begin + per);

    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
    if (vec_ok && c0 + VEC <= cols) {
        const T* col = G + c0;
        int64_t r = r_begin + warp;
        for (; r + (kUnroll - 1) * kWarps < r_end; r += kUnroll * kWarps) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                v[u] = __ldg(reinterpret_cast<const uint4*>(col + (r + u * kWarps) * ldg));
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) Elem<T>::add(v[u], acc);
        }
        for (; r < r_end; r += kWarps)
            Elem<T>::add(__ldg(reinterpret_cast<const uint4*>(col + r * ldg)), acc);
    } else {
        for (int64_t r = r_begin + warp; r < r_end; r += kWarps)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (c0 + e < cols) acc[e] += Elem<T>::one(G + r * ldg + c0 + e);
    }

    // fixed-order combine: warps of this CTA, then CTAs of the cluster
#pragma unroll
    for (int e = 0; e < VEC; ++e) part[warp][lane * VEC + e] = acc[e];
    __syncthreads();
    for (int c = threadIdx.x; c < kCols; c += kWarps * 32) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += part[w][c];
        total[c] = s;
    }
    cluster_sync();  // every CTA's total[] is written and visible to the cluster
    if (rank == 0) {
        for (int c = threadIdx.x; c < kCols; c += kWarps * 32) {
            const int64_t j = static_cast<int64_t>(blockIdx.x) * kCols + c;
            float s = 0.0f;
#pragma unroll
            for (int q = 0; q < kCluster; ++q) s += ld_shared_cluster_f32(map_to_cta(smem_u32(&total[c]), q));
            if (j < cols) out[j] = s;
        }
    }
    cluster_sync();  // the other CTAs' shared memory stays until rank 0 has read it
}

template <typename T>
cudaError_t launch_typed(const void* G, int64_t rows, int64_t cols, int64_t ldg, float* out,
                         cudaStream_t stream) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t blocks = (cols + 32 * VEC - 1) / (32 * VEC);
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int vec_ok = (reinterpret_cast<uintptr_t>(G) % 16 == 0) && (ldg % VEC == 0);
    sum_rows_kernel<T><<<dim3(static_cast<unsigned>(blocks), kCluster), kWarps * 32, 0, stream>>>(
        static_cast<const T*>(G), rows, cols, ldg, out, vec_ok);
    return cudaGetLastError();
}

}  // namespace

cudaError_t sum_rows_launch(int dtype, int64_t rows, int64_t cols, const void* G, int64_t ldg,
                            float* out, cudaStream_t stream) {
    if (dtype == DGA_F32) return launch_typed<float>(G, rows, cols, ldg, out, stream);
    if (dtype == DGA_BF16) return launch_typed<__nv_bfloat16>(G, rows, cols, ldg, out, stream);
    return launch_typed<__half>(G, rows, cols, ldg, out, stream);
}

}  // namespace dga
