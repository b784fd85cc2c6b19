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
#include <cuda.h>
#include <cudaTypedefs.h>

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

// The unique ID of the calling thread's current CUDA context (0: none, or the
// driver entry points are unavailable).  IDs are never reused, so a context
// destroyed and created again (after cudaDeviceReset, say) has a new one.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

struct ScratchEntry {
    unsigned long long ctx_id;  // context the address was looked up in
    void* ptr;
};
std::mutex g_setup_mutex;
ScratchEntry g_scratch[kda::kMaxDevices];  // per device ordinal

// Device address of the scratch on the current device.  Looked up on the first
// call in a context and again whenever the context has changed (a device
// reset reloads the library's device code, which may move the array).
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kda::kMaxDevices) return KDA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchEntry& e = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (e.ptr == nullptr || id == 0 || id != e.ctx_id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_prefill_scratch) != cudaSuccess || ptr == nullptr) return KDA_ERR_DEVICE;
        e.ptr = ptr;
        e.ctx_id = current_context_id();  // the lookup made the primary context current if none was
    }
    *out = e.ptr;
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
