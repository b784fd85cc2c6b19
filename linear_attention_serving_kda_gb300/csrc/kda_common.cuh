// kda_common.cuh -- device helpers shared by the KDA kernels (sm_103a).
//
// Per-row activations of the Kimi Delta Attention layer (ONNX Runtime GenAI
// PR #2843, "Summary of Changes": CausalConvWithState, GatedDeltaNet with
// per-key-dim decay and gate_activation='sigmoid', GatedRMSNorm(activation=
// 'sigmoid'); TensorFold issue #850, Oct 15 comment: conv window, safe or
// softplus gate, beta, q/k L2 norms, delta rule, gated output norm).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// ------------------------------------------------------------ io types

template <typename T> struct Io;
template <> struct Io<float> {
    static __device__ __forceinline__ float ld(const float* p) { return *p; }
    static __device__ __forceinline__ void st(float* p, float x) { *p = x; }
};
template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

template <typename T> __device__ __forceinline__ float ldv(const T* p) { return Io<T>::ld(p); }
template <typename T> __device__ __forceinline__ void stv(T* p, float x) { Io<T>::st(p, x); }

__device__ __forceinline__ void store_out(void* out, size_t idx, float x, int out_bf16)
{
    if (out_bf16) reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(x);
    else reinterpret_cast<float*>(out)[idx] = x;
}

// ------------------------------------------------------------ activations
// The same expressions are used by decode, verify and commit so that a
// verified row has the bits of the serially decoded one.

// e^x as 2^(x log2 e) on the special-function unit (PTX ex2.approx.ftz: a
// few ulp; inputs below about -87 give 0, the subnormal results flushed), and
// 1/x by rcp.approx.ftz: one multiply and one SFU instruction each, with no
// range handling around them.
__device__ __forceinline__ float exp_sfu(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(x, 1.44269504088896341f)));
    return y;
}
__device__ __forceinline__ float rcp_sfu(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float sigmoidf_(float x) { return rcp_sfu(__fadd_rn(1.0f, exp_sfu(-x))); }

__device__ __forceinline__ float siluf_(float x) { return __fmul_rn(x, rcp_sfu(__fadd_rn(1.0f, exp_sfu(-x)))); }

// softplus(x) = log(1 + e^x); above 20 the correction e^-x is below fp32
// resolution of x.
__device__ __forceinline__ float softplusf_(float x) { return x > 20.0f ? x : log1pf(exp_sfu(x)); }

// Per-key-dim log decay.  ea = exp(A_log_h).
__device__ __forceinline__ float log_alpha(int gate_mode, float lb, float ea, float f, float dt)
{
    float x = f + dt;
    if (gate_mode == KDA_GATE_SAFE) return lb * sigmoidf_(ea * x);
    return -ea * softplusf_(x);
}

// ------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void flag_status(int32_t* st, int bit)
{
    if (st) atomicOr(st, bit);
}

// ------------------------------------------------------------ streaming IO

__device__ __forceinline__ float4 ld_stream4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

}  // namespace kda
