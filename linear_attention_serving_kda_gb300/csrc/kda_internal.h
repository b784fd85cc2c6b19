// kda_internal.h -- host-side launch interface between the C ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

enum RecMode { REC_PREFILL = 0, REC_DECODE = 1, REC_VERIFY = 2 };

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
};

cudaError_t launch_recurrent(int mode, int io_bf16, const RecArgs& a, int units, cudaStream_t st);
cudaError_t launch_commit(int io_bf16, const CommitArgs& a, cudaStream_t st);

// Chunk kernel: returns cudaErrorNotSupported when the shape is not covered.
bool chunk_supported(const kda_params* p);
cudaError_t launch_chunk(int io_bf16, const ChunkArgs& a, cudaStream_t st);

}  // namespace kda
