// kda_chunk.cu -- chunked (WY/UT) prefill on tcgen05 tensor cores (sm_103a).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

bool chunk_supported(const kda_params* p)
{
    (void)p;
    return false;
}

cudaError_t launch_chunk(int io_bf16, const ChunkArgs& a, cudaStream_t st)
{
    (void)io_bf16; (void)a; (void)st;
    return cudaErrorNotSupported;
}

}  // namespace kda
