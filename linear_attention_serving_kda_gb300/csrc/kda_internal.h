// kda_internal.h -- host-side launch interface between the C ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/kda.h"

namespace kda {

// One-time host set-up per device (kernel attributes, capability checks) that
// several host threads may reach at once.  fn(dev) runs with the device
// current, under this object's mutex, until it has succeeded once on that
// device; afterwards callers only read an atomic flag.
constexpr int kMaxDevices = 128;
struct PerDeviceOnce {
    std::atomic<bool> done[kMaxDevices] = {};
    std::mutex m;
    template <class F> cudaError_t run(F&& fn)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(m);
        if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        e = fn(dev);
        if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
        return e;
    }
};

// REC_COMMIT_VERIFY: replay the accepted rows of the previous window's log,
// store the committed states, then verify the new window on them.
enum RecMode { REC_PREFILL = 0, REC_DECODE = 1, REC_VERIFY = 2, REC_COMMIT_VERIFY = 3 };

// Arguments of the row-recurrent kernel (decode, verify window, and the
// serial prefill used for the shapes the chunk kernel does not cover).
struct RecArgs {
    int H, D, K, gate_mode, out_bf16, num_slots, N, W, T;
    float lb, l2_eps, norm_eps, scale;
    const float* A_log;
    const float* dt_bias;
    const float* conv_w;
    const float* norm_w;
    const int32_t* cu_seqlens;
    const void* q;
    const void* k;
    const void* v;
    const void* f;
    const void* b;
    const void* g;
    const int32_t* slots;
    void* conv_state;
    float* rec_state;
    void* out;
    float* log_f;
    void* log_raw;
    int32_t* dev_status;
    // REC_COMMIT_VERIFY: rows of the previous window to commit, and its log
    const int32_t* accepted;
    const float* prev_log_f;
    const void* prev_log_raw;
};

struct CommitArgs {
    int H, D, K, num_slots, B, W;
    const int32_t* accepted;
    const int32_t* slots;
    const float* log_f;
    const void* log_raw;
    void* conv_state;
    float* rec_state;
    int32_t* dev_status;
};

// Arguments of the chunked (tensor-core) prefill.
struct ChunkArgs {
    int H, K, gate_mode, out_bf16, num_slots, N, T;
    float lb, l2_eps, norm_eps, scale;
    const float* A_log;
    const float* dt_bias;
    const float* conv_w;
    const float* norm_w;
    const int32_t* cu_seqlens;
    const void* q;
    const void* k;
    const void* v;
    const void* f;
    const void* b;
    const void* g;
    const int32_t* slots;
    void* conv_state;
    float* rec_state;
    void* out;
    int32_t* dev_status;
    int32_t* schedule;  // workspace: sequence order, longest first
    unsigned char* split_ws;  // workspace of the split (producer / chain) path, or null: fused kernel
    // Test hook (kda_debug_split_chains_only): launch the split path's chain
    // CTAs without producers, their flag waits limited to this many polls
    // (0: the normal grid and limit).
    uint32_t dbg_chains_only_polls;
    // Affine state scan (kda_prefill_scan): when nsplit > 0, units of
    // sequence index s >= nsplit are transfer runs over the rows of sequence
    // s - nsplit -- values v forced to zero, outputs to out2 -- while slots
    // stay indexed by s itself.  0: every unit is an ordinary sequence.
    int nsplit;
    void* out2;
};

cudaError_t launch_recurrent(int mode, int io_bf16, const RecArgs& a, int units, cudaStream_t st);
cudaError_t launch_commit(int io_bf16, const CommitArgs& a, cudaStream_t st);
// streaming decode at dk = dv = 128 (kda_decode.cu)
cudaError_t launch_decode_stream_d128(int io_bf16, const RecArgs& a, int units, cudaStream_t st);

// Chunk kernel: returns cudaErrorNotSupported when the shape is not covered.
bool chunk_supported(const kda_params* p);
// Few long chains (N * H <= 64 and T >= 1024 rows): the split path, whose
// workspace holds a ring of published chunk operands per chain.
bool chunk_split_wanted(const kda_params* p, int N, int T);
size_t chunk_split_bytes(int N, int H);  // flags + ring, 1 KiB aligned parts

// kda_prefill_varlen with the split path allowed or not (the built-in
// workspace of the allocation-free entry point is too small for it).
int prefill_varlen_impl(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T, const void* q,
                        const void* k, const void* v, const void* gate, const void* beta, const void* out_gate,
                        const int32_t* slots, void* conv_state, float* rec_state, void* out, void* workspace,
                        size_t ws_bytes, int32_t* dev_status, cudaStream_t stream, bool allow_split,
                        uint32_t dbg_chains_only_polls = 0);
size_t prefill_workspace_bytes(const kda_params* p, int32_t N, int32_t T, bool allow_split);
// ChunkArgs of a prefill call (every other field zero)
void fill_chunk(ChunkArgs& c, const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T, const void* q,
                const void* k, const void* v, const void* gate, const void* beta, const void* out_gate,
                const int32_t* slots, void* conv_state, float* rec_state, void* out, int32_t* dev_status);
cudaError_t launch_chunk(int io_bf16, const ChunkArgs& a, cudaStream_t st);
// Affine state scan over P segments per sequence (kda_scan.cu): a0 holds the
// call's arguments as for the fused chunk kernel; ws its workspace.
size_t prefill_scan_workspace_bytes(const kda_params* p, int N, int T, int P);
cudaError_t launch_prefill_scan(const kda_params* p, const ChunkArgs& a0, int P, unsigned char* ws, cudaStream_t st);

}  // namespace kda
