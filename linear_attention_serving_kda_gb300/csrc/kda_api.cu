// kda_api.cu -- the C ABI (include/kda.h): argument and geometry checks on the
// host, then launches on the caller's stream.  No allocation, no host sync.
//
// Geometry is rejected before anything is launched (TensorFold issue #850,
// Oct 16 comment: reject unsupported KDA head widths and tap counts before
// launch), and the gate bound is validated only in safe mode (ONNX Runtime
// GenAI PR #2843, author's review reply).
#include <cmath>
#include <cstring>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace {

using namespace kda;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int io_size(int dtype) { return dtype == KDA_DTYPE_BF16 ? 2 : 4; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
size_t align1024(size_t x) { return (x + 1023) & ~size_t(1023); }

int check_params(const kda_params* p)
{
    if (!p) return KDA_ERR_INVALID_ARGUMENT;
    if (p->num_heads <= 0 || p->num_heads > 1024) return KDA_ERR_INVALID_ARGUMENT;
    const int dk = p->head_dim_k, dv = p->head_dim_v, K = p->conv_kernel;
    if (!(dk == 32 || dk == 64 || dk == 128) || dv != dk) return KDA_ERR_UNSUPPORTED_GEOMETRY;
    if (K < 2 || K > 4) return KDA_ERR_UNSUPPORTED_GEOMETRY;
    if (p->gate_mode != KDA_GATE_SOFTPLUS && p->gate_mode != KDA_GATE_SAFE) return KDA_ERR_INVALID_ARGUMENT;
    if (p->gate_mode == KDA_GATE_SAFE && !(std::isfinite(p->gate_lower_bound) && p->gate_lower_bound < 0.0f))
        return KDA_ERR_INVALID_BOUND;
    if (!(std::isfinite(p->l2_eps) && p->l2_eps >= 0.0f)) return KDA_ERR_INVALID_ARGUMENT;
    if (!(std::isfinite(p->norm_eps) && p->norm_eps >= 0.0f)) return KDA_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(p->scale)) return KDA_ERR_INVALID_ARGUMENT;
    if (p->io_dtype != KDA_DTYPE_F32 && p->io_dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (p->out_dtype != KDA_DTYPE_F32 && p->out_dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (p->num_slots <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!p->A_log || !p->dt_bias || !p->conv_weight) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(p->A_log) || !aligned16(p->dt_bias) || !aligned16(p->conv_weight)) return KDA_ERR_INVALID_ARGUMENT;
    if (p->norm_weight && !aligned16(p->norm_weight)) return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
}

// Every pointer in the list must be non-null and 16-byte aligned.
int check_ptrs(std::initializer_list<const void*> ps)
{
    for (const void* x : ps)
        if (!x || !aligned16(x)) return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
}

int check_opt(const void* x) { return (x && !aligned16(x)) ? KDA_ERR_INVALID_ARGUMENT : KDA_OK; }

// The library is built for sm_103a only; remember the answer per device
// (the set-up object records only a successful check; -1 marks another GPU).
int check_device()
{
    static PerDeviceOnce once;
    static std::atomic<signed char> ok[kMaxDevices];  // 0 unknown, 1 yes, -1 no
    int dev = 0;
    cudaError_t e = once.run([&](int d) {
        int major = 0, minor = 0;
        cudaError_t r = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d);
        if (r == cudaSuccess) ok[d].store((major == 10 && minor == 3) ? 1 : -1, std::memory_order_relaxed);
        return r;
    });
    if (e != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_DEVICE;
    return ok[dev].load(std::memory_order_relaxed) == 1 ? KDA_OK : KDA_ERR_DEVICE;
}

void fill_common(RecArgs& a, const kda_params* p)
{
    std::memset(&a, 0, sizeof(a));
    a.H = p->num_heads;
    a.D = p->head_dim_k;
    a.K = p->conv_kernel;
    a.gate_mode = p->gate_mode;
    a.out_bf16 = p->out_dtype == KDA_DTYPE_BF16;
    a.num_slots = p->num_slots;
    a.lb = p->gate_lower_bound;
    a.l2_eps = p->l2_eps;
    a.norm_eps = p->norm_eps;
    a.scale = p->scale;
    a.A_log = p->A_log;
    a.dt_bias = p->dt_bias;
    a.conv_w = p->conv_weight;
    a.norm_w = p->norm_weight;
}

size_t log_float_bytes(const kda_params* p, int32_t B, int32_t W)
{
    return align256((size_t)B * W * p->num_heads * (2 * (size_t)p->head_dim_k + p->head_dim_v) * sizeof(float));
}

}  // namespace

extern "C" {

KDA_API int kda_abi_version(void) { return 100; }

KDA_API const char* kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
    case KDA_ERR_UNSUPPORTED_GEOMETRY: return "KDA_ERR_UNSUPPORTED_GEOMETRY";
    case KDA_ERR_INVALID_BOUND: return "KDA_ERR_INVALID_BOUND";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_LAUNCH: return "KDA_ERR_LAUNCH";
    case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
    default: return "KDA_ERR_UNKNOWN";
    }
}

}  // extern "C"

namespace kda {

size_t prefill_workspace_bytes(const kda_params* p, int32_t N, int32_t T, bool allow_split)
{
    if (check_params(p) != KDA_OK || N < 0 || T < 0) return 0;
    if (!chunk_supported(p)) return 0;
    // the chunk kernel's longest-first schedule: one int32 per sequence
    const size_t sched = align256((size_t)(N + 1) * sizeof(int32_t));
    if (allow_split && chunk_split_wanted(p, N, T)) {
        size_t b = align1024(sched) + chunk_split_bytes(N, p->num_heads);
        // gates whose per-row log-decay is not bounded by -5: each chain's
        // chunk list (a count, up to T chunk starts, the end, the first cut
        // chunk) after the ring
        if (!(p->gate_mode == KDA_GATE_SAFE && p->gate_lower_bound >= -5.0f))
            b += align1024((size_t)N * p->num_heads * ((size_t)T + 3) * sizeof(int32_t));
        // the chains' outputs before the epilogue: fp32 [T][H][dv]
        b += align1024((size_t)T * p->num_heads * p->head_dim_v * sizeof(float));
        return b;
    }
    return sched;
}

}  // namespace kda

extern "C" {

KDA_API size_t kda_prefill_workspace_bytes(const kda_params* p, int32_t N, int32_t T)
{
    return prefill_workspace_bytes(p, N, T, true);
}

KDA_API size_t kda_verify_log_bytes(const kda_params* p, int32_t B, int32_t W)
{
    if (check_params(p) != KDA_OK || B < 0 || W < 0) return 0;
    const size_t conv_dim = (size_t)p->num_heads * (2 * p->head_dim_k + p->head_dim_v);
    return log_float_bytes(p, B, W) + align256((size_t)B * W * conv_dim * io_size(p->io_dtype));
}

}  // extern "C"

int kda::prefill_varlen_impl(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T,
                             const void* q, const void* k, const void* v, const void* gate, const void* beta,
                             const void* out_gate, const int32_t* slots, void* conv_state, float* rec_state,
                             void* out, void* workspace, size_t ws_bytes, int32_t* dev_status,
                             cudaStream_t stream, bool allow_split, uint32_t dbg_chains_only_polls)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (N < 0 || T < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    if ((rc = check_ptrs({cu_seqlens, conv_state, rec_state})) != KDA_OK) return rc;
    if (T > 0 && (rc = check_ptrs({q, k, v, gate, beta, out})) != KDA_OK) return rc;
    if ((rc = check_opt(out_gate)) != KDA_OK || (rc = check_opt(slots)) != KDA_OK) return rc;
    const size_t need = prefill_workspace_bytes(p, N, T, allow_split);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace))) return KDA_ERR_WORKSPACE;
    if ((rc = check_device()) != KDA_OK) return rc;

    if (chunk_supported(p)) {
        ChunkArgs c;
        fill_chunk(c, p, cu_seqlens, N, T, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state, out,
                   dev_status);
        c.schedule = static_cast<int32_t*>(workspace);
        if (allow_split && chunk_split_wanted(p, N, T))
            c.split_ws = static_cast<unsigned char*>(workspace) + align1024(align256((size_t)(N + 1) * sizeof(int32_t)));
        c.dbg_chains_only_polls = dbg_chains_only_polls;
        return launch_chunk(p->io_dtype == KDA_DTYPE_BF16, c, stream) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
    }
    RecArgs a;
    fill_common(a, p);
    a.N = N;
    a.W = 1;
    a.T = T;
    a.cu_seqlens = cu_seqlens;
    a.q = q; a.k = k; a.v = v; a.f = gate; a.b = beta; a.g = out_gate;
    a.slots = slots;
    a.conv_state = conv_state;
    a.rec_state = rec_state;
    a.out = out;
    a.dev_status = dev_status;
    return launch_recurrent(REC_PREFILL, p->io_dtype == KDA_DTYPE_BF16, a, N * p->num_heads, stream) == cudaSuccess
               ? KDA_OK : KDA_ERR_LAUNCH;
}

void kda::fill_chunk(ChunkArgs& c, const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T,
                     const void* q, const void* k, const void* v, const void* gate, const void* beta,
                     const void* out_gate, const int32_t* slots, void* conv_state, float* rec_state, void* out,
                     int32_t* dev_status)
{
    {
        std::memset(&c, 0, sizeof(c));
        c.H = p->num_heads;
        c.K = p->conv_kernel;
        c.gate_mode = p->gate_mode;
        c.out_bf16 = p->out_dtype == KDA_DTYPE_BF16;
        c.num_slots = p->num_slots;
        c.N = N;
        c.T = T;
        c.lb = p->gate_lower_bound;
        c.l2_eps = p->l2_eps;
        c.norm_eps = p->norm_eps;
        c.scale = p->scale;
        c.A_log = p->A_log;
        c.dt_bias = p->dt_bias;
        c.conv_w = p->conv_weight;
        c.norm_w = p->norm_weight;
        c.cu_seqlens = cu_seqlens;
        c.q = q; c.k = k; c.v = v; c.f = gate; c.b = beta; c.g = out_gate;
        c.slots = slots;
        c.conv_state = conv_state;
        c.rec_state = rec_state;
        c.out = out;
        c.dev_status = dev_status;
    }
}

extern "C" {

KDA_API int kda_prefill_varlen(const kda_params* p, const int32_t* cu_seqlens, int32_t N,
                               int32_t T, const void* q, const void* k, const void* v,
                               const void* gate, const void* beta, const void* out_gate,
                               const int32_t* slots, void* conv_state, float* rec_state,
                               void* out, void* workspace, size_t ws_bytes,
                               int32_t* dev_status, cudaStream_t stream)
{
    return prefill_varlen_impl(p, cu_seqlens, N, T, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state,
                               out, workspace, ws_bytes, dev_status, stream, true);
}

KDA_API size_t kda_prefill_scan_workspace_bytes(const kda_params* p, int32_t N, int32_t T, int32_t segments)
{
    if (check_params(p) != KDA_OK || N < 0 || T < 0 || segments < 1 || segments > KDA_SCAN_MAX_SEGMENTS) return 0;
    if (!chunk_supported(p)) return 0;
    return prefill_scan_workspace_bytes(p, N, T, segments);
}

KDA_API int kda_prefill_scan(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T, const void* q,
                             const void* k, const void* v, const void* gate, const void* beta, const void* out_gate,
                             const int32_t* slots, void* conv_state, float* rec_state, void* out, void* workspace,
                             size_t ws_bytes, int32_t segments, int32_t* dev_status, cudaStream_t stream)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (N < 0 || T < 0 || segments < 1 || segments > KDA_SCAN_MAX_SEGMENTS) return KDA_ERR_INVALID_ARGUMENT;
    if (!chunk_supported(p)) return KDA_ERR_UNSUPPORTED_GEOMETRY;
    if (N == 0) return KDA_OK;
    if ((rc = check_ptrs({cu_seqlens, conv_state, rec_state})) != KDA_OK) return rc;
    if (T > 0 && (rc = check_ptrs({q, k, v, gate, beta, out})) != KDA_OK) return rc;
    if ((rc = check_opt(out_gate)) != KDA_OK || (rc = check_opt(slots)) != KDA_OK) return rc;
    const size_t need = prefill_scan_workspace_bytes(p, N, T, segments);
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    if ((rc = check_device()) != KDA_OK) return rc;
    ChunkArgs c;
    fill_chunk(c, p, cu_seqlens, N, T, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state, out, dev_status);
    return launch_prefill_scan(p, c, segments, static_cast<unsigned char*>(workspace), stream) == cudaSuccess
               ? KDA_OK : KDA_ERR_LAUNCH;
}

KDA_API int kda_debug_split_chains_only(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T,
                                        const void* q, const void* k, const void* v, const void* gate,
                                        const void* beta, const void* out_gate, const int32_t* slots,
                                        void* conv_state, float* rec_state, void* out, void* workspace,
                                        size_t ws_bytes, int32_t* dev_status, uint32_t poll_limit,
                                        cudaStream_t stream)
{
    if (!chunk_supported(p) || !chunk_split_wanted(p, N, T) || poll_limit == 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!(p->gate_mode == KDA_GATE_SAFE && p->gate_lower_bound >= -5.0f)) return KDA_ERR_INVALID_ARGUMENT;
    return prefill_varlen_impl(p, cu_seqlens, N, T, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state,
                               out, workspace, ws_bytes, dev_status, stream, true, poll_limit);
}

namespace {
__global__ void activations_kernel(int which, const float* x, float* y, int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float v = x[i];
        y[i] = which == KDA_ACT_EXP ? kda::exp_sfu(v)
             : which == KDA_ACT_RCP ? kda::rcp_sfu(v)
             : which == KDA_ACT_SIGMOID ? kda::sigmoidf_(v)
             : kda::siluf_(v);
    }
}
}  // namespace

KDA_API int kda_debug_activations(int32_t which, const float* x, float* y, int32_t n, cudaStream_t stream)
{
    if (which < KDA_ACT_EXP || which > KDA_ACT_SILU || n < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (n == 0) return KDA_OK;
    int rc = check_ptrs({x, y});
    if (rc != KDA_OK) return rc;
    if ((rc = check_device()) != KDA_OK) return rc;
    activations_kernel<<<(n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024, 256, 0, stream>>>(which, x, y, n);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

KDA_API int kda_decode(const kda_params* p, int32_t B, const void* q, const void* k,
                       const void* v, const void* gate, const void* beta,
                       const void* out_gate, const int32_t* slots, void* conv_state,
                       float* rec_state, void* out, int32_t* dev_status, cudaStream_t stream)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (B < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (B == 0) return KDA_OK;
    if ((rc = check_ptrs({q, k, v, gate, beta, conv_state, rec_state, out})) != KDA_OK) return rc;
    if ((rc = check_opt(out_gate)) != KDA_OK || (rc = check_opt(slots)) != KDA_OK) return rc;
    if ((rc = check_device()) != KDA_OK) return rc;
    RecArgs a;
    fill_common(a, p);
    a.N = B;
    a.W = 1;
    a.T = B;
    a.q = q; a.k = k; a.v = v; a.f = gate; a.b = beta; a.g = out_gate;
    a.slots = slots;
    a.conv_state = conv_state;
    a.rec_state = rec_state;
    a.out = out;
    a.dev_status = dev_status;
    return launch_recurrent(REC_DECODE, p->io_dtype == KDA_DTYPE_BF16, a, B * p->num_heads, stream) == cudaSuccess
               ? KDA_OK : KDA_ERR_LAUNCH;
}

KDA_API int kda_verify_window(const kda_params* p, int32_t B, int32_t W, const void* q,
                              const void* k, const void* v, const void* gate,
                              const void* beta, const void* out_gate,
                              const int32_t* slots, const void* conv_state,
                              const float* rec_state, void* log, void* out,
                              int32_t* dev_status, cudaStream_t stream)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (B < 0 || W < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (B == 0 || W == 0) return KDA_OK;
    if ((rc = check_ptrs({q, k, v, gate, beta, conv_state, rec_state, log, out})) != KDA_OK) return rc;
    if ((rc = check_opt(out_gate)) != KDA_OK || (rc = check_opt(slots)) != KDA_OK) return rc;
    if ((rc = check_device()) != KDA_OK) return rc;
    RecArgs a;
    fill_common(a, p);
    a.N = B;
    a.W = W;
    a.T = B * W;
    a.q = q; a.k = k; a.v = v; a.f = gate; a.b = beta; a.g = out_gate;
    a.slots = slots;
    a.conv_state = const_cast<void*>(conv_state);
    a.rec_state = const_cast<float*>(rec_state);
    a.out = out;
    a.log_f = static_cast<float*>(log);
    a.log_raw = static_cast<char*>(log) + log_float_bytes(p, B, W);
    a.dev_status = dev_status;
    return launch_recurrent(REC_VERIFY, p->io_dtype == KDA_DTYPE_BF16, a, B * p->num_heads, stream) == cudaSuccess
               ? KDA_OK : KDA_ERR_LAUNCH;
}

KDA_API int kda_commit_verify(const kda_params* p, int32_t B, int32_t W, const int32_t* accepted,
                              const void* log_prev, const void* q, const void* k, const void* v,
                              const void* gate, const void* beta, const void* out_gate,
                              const int32_t* slots, void* conv_state, float* rec_state, void* log,
                              void* out, int32_t* dev_status, cudaStream_t stream)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (B < 0 || W < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (B == 0 || W == 0) return KDA_OK;
    if ((rc = check_ptrs({accepted, log_prev, q, k, v, gate, beta, conv_state, rec_state, log, out})) != KDA_OK)
        return rc;
    if ((rc = check_opt(out_gate)) != KDA_OK || (rc = check_opt(slots)) != KDA_OK) return rc;
    if ((rc = check_device()) != KDA_OK) return rc;
    RecArgs a;
    fill_common(a, p);
    a.N = B;
    a.W = W;
    a.T = B * W;
    a.q = q; a.k = k; a.v = v; a.f = gate; a.b = beta; a.g = out_gate;
    a.slots = slots;
    a.conv_state = conv_state;
    a.rec_state = rec_state;
    a.out = out;
    a.log_f = static_cast<float*>(log);
    a.log_raw = static_cast<char*>(log) + log_float_bytes(p, B, W);
    a.accepted = accepted;
    a.prev_log_f = static_cast<const float*>(log_prev);
    a.prev_log_raw = static_cast<const char*>(log_prev) + log_float_bytes(p, B, W);
    a.dev_status = dev_status;
    return launch_recurrent(REC_COMMIT_VERIFY, p->io_dtype == KDA_DTYPE_BF16, a, B * p->num_heads, stream) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_LAUNCH;
}

KDA_API int kda_commit(const kda_params* p, int32_t B, int32_t W, const int32_t* accepted,
                       const int32_t* slots, const void* log, void* conv_state,
                       float* rec_state, int32_t* dev_status, cudaStream_t stream)
{
    int rc = check_params(p);
    if (rc != KDA_OK) return rc;
    if (B < 0 || W < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (B == 0 || W == 0) return KDA_OK;
    if ((rc = check_ptrs({accepted, log, conv_state, rec_state})) != KDA_OK) return rc;
    if ((rc = check_opt(slots)) != KDA_OK) return rc;
    if ((rc = check_device()) != KDA_OK) return rc;
    CommitArgs a;
    std::memset(&a, 0, sizeof(a));
    a.H = p->num_heads;
    a.D = p->head_dim_k;
    a.K = p->conv_kernel;
    a.num_slots = p->num_slots;
    a.B = B;
    a.W = W;
    a.accepted = accepted;
    a.slots = slots;
    a.log_f = static_cast<const float*>(log);
    a.log_raw = static_cast<const char*>(log) + log_float_bytes(p, B, W);
    a.conv_state = conv_state;
    a.rec_state = rec_state;
    a.dev_status = dev_status;
    return launch_commit(p->io_dtype == KDA_DTYPE_BF16, a, stream) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // extern "C"
