// kda_prefill_static.cu -- a prefill entry point that allocates nothing.
//
// kda_prefill_varlen asks its caller for a device workspace (the chunk
// kernel's longest-first sequence order).  Some callers cannot provide one:
// code running inside an allocator-free runtime, a plugin that may not touch
// the host process's memory pools, or a serving loop that must not call
// cudaMalloc at all once it is running.  For them this variant keeps the
// workspace in a fixed array in the library's own device memory.
//
// That array lives for as long as the library is loaded, on every GPU the
// library is used on.  All calls share it and it keeps whatever the previous
// call left there; the chunk kernel's scheduler rewrites every entry it reads,
// so nothing has to be cleared between calls.  Two calls whose kernels run at
// the same time on one GPU (different streams, no ordering between them)
// would race on the array and must not be issued.
#include <mutex>

#include "kda_internal.h"

namespace {

// Capacity of the built-in workspace: the prefill needs (N + 1) int32 values
// rounded up to 256 bytes, so up to 65535 sequences per call.
constexpr size_t kStaticWorkspaceBytes = 256 * 1024;

// The scratch itself (device memory of every GPU that loads the library).
// In host code this name is only a host-side handle: the kernel must be given
// the device address that cudaGetSymbolAddress returns for it.
static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticWorkspaceBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[128];  // per device ordinal, filled on first use

// Device address of the scratch on the current device (set up once per device).
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return KDA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_prefill_scratch) != cudaSuccess || ptr == nullptr) return KDA_ERR_DEVICE;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

KDA_API size_t kda_prefill_static_workspace_capacity(void) { return kStaticWorkspaceBytes; }

KDA_API int kda_prefill_varlen_static_ws(const kda_params* p, const int32_t* cu_seqlens, int32_t N,
                                         int32_t T, const void* q, const void* k, const void* v,
                                         const void* gate, const void* beta, const void* out_gate,
                                         const int32_t* slots, void* conv_state, float* rec_state,
                                         void* out, int32_t* dev_status, cudaStream_t stream)
{
    // the fused chunk path only: the split path's ring does not fit the built-in workspace
    const size_t need = kda::prefill_workspace_bytes(p, N, T, false);
    if (need > kStaticWorkspaceBytes) return KDA_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&ws);
        if (rc != KDA_OK) return rc;
    }
    return kda::prefill_varlen_impl(p, cu_seqlens, N, T, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state,
                                    out, ws, need > 0 ? kStaticWorkspaceBytes : 0, dev_status, stream, false);
}

}  // extern "C"
