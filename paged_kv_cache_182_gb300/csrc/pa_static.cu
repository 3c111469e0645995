// pa_static.cu -- pa_decode_static_workspace: decode attention with the split
// scratch taken from a fixed array inside the library, for callers that are
// not allowed to allocate device memory (see include/pa_decode.h).
//
// The array lives in device global memory of every GPU that loads this
// library, for the life of the process.  Host code never touches it by name
// except to ask the runtime for its device address: in host code the symbol is
// only a stand-in, and handing it to a kernel would read the wrong memory.

#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
int static_workspace_address(void** addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p)
            return PA_ERR_CUDA;
        g_static_addr[dev] = p;
    }
    *addr = g_static_addr[dev];
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
