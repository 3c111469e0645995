// pa_static.cu -- pa_decode_static_workspace: decode attention with the split
// scratch taken from a fixed array inside the library, for callers that are
// not allowed to allocate device memory (see include/pa_decode.h).
//
// The array lives in device global memory of every GPU that loads this
// library, for the life of the process.  Host code never touches it by name
// except to ask the runtime for its device address: in host code the symbol is
// only a stand-in, and handing it to a kernel would read the wrong memory.

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The array's device address belongs to the context that loaded the module:
// a device reset, or another context made current on the same device, loads
// the module again at another address.  So each cached address is tagged with
// the unique id of the context it was looked up in (cuCtxGetId, never reused
// within a process), and a call made under another context looks it up again.
struct StaticAddr {
    unsigned long long ctx_id;  // 0 = nothing cached
    void* addr;
};
std::mutex g_static_mutex;
StaticAddr g_static_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name)
{
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(ptr);
}

// Unique id of the context current on this thread, 0 when there is none (or
// the driver cannot say): 0 is never cached, so such calls always look up.
unsigned long long current_context_id()
{
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array on the current device and context.  Looked up
// with cudaGetSymbolAddress the first time a context asks, then cached.
int static_workspace_address(void** addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_static_mutex);
    StaticAddr& c = g_static_addr[dev];
    if (id != 0 && c.ctx_id == id && c.addr) {
        *addr = c.addr;
        return PA_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p)
        return PA_ERR_CUDA;
    // the lookup binds the device's primary context when none was current
    c.ctx_id = id != 0 ? id : current_context_id();
    c.addr = p;
    *addr = p;
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, const int32_t* seq_lens,
                                          const void* k_new, const void* v_new, void* out,
                                          float scale, int H, int KV, int D, int BLOCK, int NQ,
                                          int causal, const pa_opts* opts, void* stream)
{
    if (!opts)
        return PA_ERR_NULL_POINTER;
    // 0 for arguments pa_decode itself rejects; those errors come from pa_decode.
    const size_t need = pa_workspace_bytes(opts->batch, H, KV, D, NQ, opts->partitions);
    if (need > PA_STATIC_WORKSPACE_BYTES)
        return PA_ERR_STATIC_LIMIT;
    pa_opts local = *opts;
    local.workspace = nullptr;
    local.workspace_bytes = 0;
    local.merge_kernel = 1;  // no split counters: nothing in the array must start at zero
    if (need > 0) {
        void* addr = nullptr;
        const int rc = static_workspace_address(&addr);
        if (rc != PA_OK)
            return rc;
        local.workspace = addr;
        local.workspace_bytes = PA_STATIC_WORKSPACE_BYTES;
    }
    return pa_decode(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, out, scale, H, KV,
                     D, BLOCK, NQ, causal, &local, stream);
}
