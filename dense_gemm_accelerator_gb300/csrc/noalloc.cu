// noalloc.cu -- INT8 x INT8 -> INT32 GEMM for callers that cannot allocate
// device memory.
//
// The regular INT8 path needs a scratch buffer (the operands re-encoded as
// bf16, each in its own layout) that the caller passes in as `workspace`.  Some callers have
// no way to provide one: a plugin that is handed only its input and output
// buffers by a host application, a serving engine that reserves all device
// memory when it starts and refuses allocations afterwards, or a
// latency-critical loop that cannot afford cudaMalloc's implicit
// synchronisation of the whole device.  dga_gemm_i8_noalloc serves them with
// a fixed scratch area compiled into the library instead.
//
// The scratch is a file-scope __device__ array of DGA_NOALLOC_SCRATCH_BYTES
// (72 MiB).  Every GPU on which this entry point is used holds it until the
// process exits.  All calls share it and it keeps the last call's contents;
// nothing in it needs to start at zero, because each call rewrites every byte
// it later reads (the repack writes whole padded rows).  Calls that overlap on
// the GPU (two streams, or two host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "dga_internal.h"

namespace {

constexpr size_t kScratchBytes = 72ull << 20;
static_assert(kScratchBytes == DGA_NOALLOC_SCRATCH_BYTES, "header and library disagree");

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_scratch[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// The array's name in host code is only a host-side handle; kernels need its
// device address, which is looked up once per device with that device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_scratch[dev] = p;
    });
    *out = g_scratch[dev];
    return g_scratch_err[dev];
}

// dga_gemm_ex reports a bad argument as -(its position there); this entry
// point has fewer arguments, so map those positions onto its own.
int remap_argument_error(int st) {
    if (st >= 0) return st;
    switch (-st) {
    case 3: return -1;   // layout_b
    case 4: return -2;   // M
    case 5: return -3;   // N
    case 6: return -4;   // K
    case 7: return -5;   // alpha
    case 8: return -6;   // A
    case 9: return -7;   // lda
    case 10: return -8;  // B
    case 11: return -9;  // ldb
    case 12: return -10; // beta
    case 13: return -11; // C
    case 14: return -12; // ldc
    default: return st;
    }
}

}  // namespace

extern "C" int dga_gemm_i8_noalloc(dga_layout layout_b, int64_t M, int64_t N, int64_t K,
                                   const int32_t* alpha, const int8_t* A, int64_t lda,
                                   const int8_t* B, int64_t ldb, const int32_t* beta, int32_t* C,
                                   int64_t ldc, dga_stream_t stream) {
    // A call that would not fit the fixed scratch is refused before anything
    // is enqueued (invalid sizes make the query return 0; dga_gemm_ex then
    // reports them).
    const size_t need = dga_gemm_workspace_size(DGA_I8, DGA_I32, layout_b, M, N, K, lda, ldb, ldc,
                                                DGA_PATH_TCGEN05);
    if (need > kScratchBytes) return DGA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) return dga::note_cuda_error(e);
    }
    const bool product = K > 0 && alpha != nullptr && *alpha != 0;
    const int st = dga_gemm_ex(DGA_I8, DGA_I32, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C,
                               ldc, scratch, scratch ? kScratchBytes : 0,
                               product ? DGA_PATH_TCGEN05 : DGA_PATH_AUTO, stream);
    return remap_argument_error(st);
}
