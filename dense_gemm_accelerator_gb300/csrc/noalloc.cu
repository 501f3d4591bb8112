// noalloc.cu -- INT8 x INT8 -> INT32 GEMM for callers that cannot allocate
// device memory.
//
// The regular INT8 path needs a scratch buffer (the operands re-encoded as
// bf16, both K-major) that the caller passes in as `workspace`.  Some callers have
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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dga_internal.h"

namespace {

constexpr size_t kScratchBytes = 72ull << 20;
static_assert(kScratchBytes == DGA_NOALLOC_SCRATCH_BYTES, "header and library disagree");

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// In host code the array's name is only a host-side handle; kernels need its
// device address.  That address belongs to the CUDA context the library's
// module is loaded in (normally a device's primary context), so it is looked
// up with the device current, once per context, and cached under the
// context's ID: unlike the context handle, which a context created after
// cudaDeviceReset may reuse, the ID is never given to a second context in a
// process.  A reset or another context therefore gets a fresh lookup instead
// of a stale address.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return fns;
}

// The ID of the current context, or false when there is none yet or the
// driver cannot say.
bool current_context_id(unsigned long long* id) {
    const DriverFns& f = driver_fns();
    if (!f.get_current || !f.get_id) return false;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return f.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kCacheSlots = 64;
std::mutex g_cache_mutex;
unsigned long long g_cache_id[kCacheSlots];
void* g_cache_addr[kCacheSlots];
int g_cache_used = 0;
int g_cache_next = 0;  // once all slots are taken: the oldest entry, replaced next

cudaError_t scratch_address(void** out) {
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (have_id) {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        for (int i = 0; i < g_cache_used; ++i)
            if (g_cache_id[i] == id) {
                *out = g_cache_addr[i];
                return cudaSuccess;
            }
    }
    // Not seen yet (or no context made current so far: this call creates the
    // device's primary context).  Look the address up with the device current.
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (current_context_id(&id)) {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        int slot;
        if (g_cache_used < kCacheSlots) {
            slot = g_cache_used++;
        } else {  // every slot taken: the oldest entry makes room
            slot = g_cache_next;
            g_cache_next = (g_cache_next + 1) % kCacheSlots;
        }
        g_cache_id[slot] = id;
        g_cache_addr[slot] = p;
    }
    *out = p;
    return cudaSuccess;
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
    // A call whose repacked operands would not fit the fixed scratch is
    // refused before anything is enqueued (invalid sizes make the query return
    // 0; dga_gemm_ex then reports them).  Only the bytes the call cannot run
    // without count here, not the optional ones the public size query adds
    // for the split last waves of other paths.
    const size_t need = dga::workspace_required_bytes(DGA_I8, DGA_I32, DGA_ROW_MAJOR, layout_b, M, N,
                                                      K, lda, ldb, ldc, DGA_PATH_TCGEN05);
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
