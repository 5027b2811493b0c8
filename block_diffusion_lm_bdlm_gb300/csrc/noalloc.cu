// noalloc.cu - bdlm_attn_fwd_noalloc: the forward without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: plugins hosted by a framework or server that owns every device
// allocation and hands out no allocator, and real-time services that forbid
// allocation after start-up. They still own and pass q, k, v, o
// and lse; the forward's own scratch (the tile table, the work counter and
// the device error word) lives here instead, in a fixed array that every GPU
// which loads this library holds until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "bdlm.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB: enough for ~2.5 M rows

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_mu;
struct Cached {
    CUcontext ctx;  // the context the address belongs to
    void* addr;     // device address of g_fwd_scratch in that context
};
Cached g_cache[128] = {};

// cuCtxGetCurrent through the runtime's driver entry-point query, so that the
// library keeps no link-time dependency on the driver library (it loads, and
// its host-side checks run, on machines without a GPU driver).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CUcontext current_context() {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return nullptr;
        fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    CUcontext c = nullptr;
    if (fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the scratch on the current device. The name
// g_fwd_scratch in host code is only a host-side stand-in; the address a
// kernel may use comes from cudaGetSymbolAddress, taken with the device
// current. It is cached per device together with the context it was taken
// in, and looked up again when that context changes (after a device reset
// the runtime loads the module into a new primary context, at a new address).
int scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return BDLM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    Cached& c = g_cache[dev];
    CUcontext ctx = current_context();
    if (!c.addr || !ctx || ctx != c.ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return BDLM_ERR_CUDA;
        c.addr = p;
        c.ctx = current_context();  // the lookup makes the runtime's context current if it was not
    }
    *out = c.addr;
    return BDLM_OK;
}

}  // namespace

namespace bdlm {
int noalloc_scratch(void** out) { return scratch_on_current_device(out); }
}  // namespace bdlm

extern "C" BDLM_API int bdlm_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                              int64_t L, int32_t block, int32_t heads, int32_t kv_heads,
                                              int32_t head_dim, const int32_t* cu_seqlens, int32_t n_docs,
                                              float softmax_scale, const bdlm_partial* part,
                                              bdlm_stream_t stream) {
    const size_t need = bdlm_attn_fwd_workspace_bytes(L, heads, head_dim, cu_seqlens ? n_docs : 1);
    if (need == 0) return BDLM_ERR_INVALID_ARG;
    if (need > kScratchBytes) return BDLM_ERR_WORKSPACE;  // beyond the fixed scratch: use bdlm_attn_fwd
    void* ws = nullptr;
    const int st = scratch_on_current_device(&ws);
    if (st != BDLM_OK) return st;
    return bdlm_attn_fwd(q, k, v, o, lse, L, block, heads, kv_heads, head_dim, cu_seqlens, n_docs, softmax_scale,
                         part, ws, kScratchBytes, stream);
}
