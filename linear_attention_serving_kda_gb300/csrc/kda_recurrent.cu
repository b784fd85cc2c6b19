// kda_recurrent.cu -- row-recurrent KDA kernels for sm_103a: decode rows,
// verify windows, the serial prefill, and the verify commit.
//
// One CTA of 256 threads owns one (sequence, head) unit.  The fp32 dk x dv
// state lives in registers for the whole call: warp w holds rows
// [w*D/8, (w+1)*D/8) and lane l holds columns [l*D/32, (l+1)*D/32), so each
// warp streams whole 128-float rows (coalesced, 16-byte vector loads) and
// the two key-dim reductions per row (S'^T k and S^T q) are an in-register
// partial over the warp's rows followed by a fixed-order sum over the 8
// warps in shared memory.
//
// Decode, verify and commit run the same per-element expressions in the same
// order -- S' = alpha * S (rounded), then S = fma(k, u, S') -- with the same
// thread-to-element map and the same reduction trees, so a verified row has
// the bits of a decoded row and a committed state the bits of serial decode
// (TensorFold issue #850, Oct 15 comment: a window logs each row's decay,
// normalized key and update, and the replay gives the bits of rows decoded
// one at a time; Oct 19 comment: preserve rounding, reduction order, replay).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int REC_THREADS = 256;
constexpr int REC_WARPS = REC_THREADS / 32;

template <int D> struct RecShape {
    static constexpr int CPT = D / 32;        // state columns per lane
    static constexpr int RPW = D / REC_WARPS; // state rows per warp
};

template <int D> struct RecSmem {
    float win[4][3 * D];      // ring of the last 4 raw conv rows (this head's q|k|v channels)
    float cw[3 * D][4];       // conv taps
    float dtb[D];             // dt_bias of this head
    float act[3 * D];         // post-SiLU q', k', v'
    float qn[D], kn[D], alpha[D], u[D], fr[D];
    float red[REC_WARPS][D];  // cross-warp partial sums
    float scal[8];
};

__device__ __forceinline__ int ring(int x) { return x & 3; }

// Global channel of local channel c (q | k | v of head h) in the conv layout.
template <int D> __device__ __forceinline__ int conv_channel(int c, int h, int H)
{
    if (c < D) return h * D + c;
    if (c < 2 * D) return H * D + h * D + (c - D);
    return 2 * H * D + h * D + (c - 2 * D);
}

template <int D> __device__ __forceinline__ void load_tile(const float* Sg, int r0, int c0,
                                                           float (&s)[RecShape<D>::RPW][RecShape<D>::CPT])
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const float* p = Sg + (size_t)(r0 + rr) * D + c0;
        if constexpr (CPT == 4) {
            float4 x = ld_stream4(p);
            s[rr][0] = x.x; s[rr][1] = x.y; s[rr][2] = x.z; s[rr][3] = x.w;
        } else if constexpr (CPT == 2) {
            float2 x = __ldcs(reinterpret_cast<const float2*>(p));
            s[rr][0] = x.x; s[rr][1] = x.y;
        } else {
            s[rr][0] = __ldcs(p);
        }
    }
}

template <int D> __device__ __forceinline__ void store_tile(float* Sg, int r0, int c0,
                                                            const float (&s)[RecShape<D>::RPW][RecShape<D>::CPT])
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        float* p = Sg + (size_t)(r0 + rr) * D + c0;
        if constexpr (CPT == 4) {
            st_stream4(p, make_float4(s[rr][0], s[rr][1], s[rr][2], s[rr][3]));
        } else if constexpr (CPT == 2) {
            __stcs(reinterpret_cast<float2*>(p), make_float2(s[rr][0], s[rr][1]));
        } else {
            __stcs(p, s[rr][0]);
        }
    }
}

template <int D, typename IO, int MODE>
__global__ void __launch_bounds__(REC_THREADS, 2) kda_recurrent_kernel(const RecArgs a)
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    __shared__ RecSmem<D> sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, K = a.K;
    const int seq = blockIdx.x / H, h = blockIdx.x % H;
    const int conv_dim = H * 3 * D;

    const int slot = a.slots ? a.slots[seq] : seq;
    if (slot < 0) return;  // padding sequence: nothing to do
    if (slot >= a.num_slots) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    int row0, L;
    if (MODE == REC_PREFILL) {
        const int s0 = a.cu_seqlens[seq], s1 = a.cu_seqlens[seq + 1];
        if (s0 < 0 || s1 < s0 || s1 > a.T) {
            if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SEQLENS);
            return;
        }
        row0 = s0;
        L = s1 - s0;
        if (L == 0) return;  // zero-length sequence: states unchanged
    } else if (MODE == REC_DECODE) {
        row0 = seq;
        L = 1;
    } else {
        row0 = seq * a.W;
        L = a.W;
    }

    // State tile first: its HBM stream overlaps the row preparation below.
    float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
    const int r0 = warp * RPW, c0 = lane * CPT;
    float s[RPW][CPT];
    load_tile<D>(Sg, r0, c0, s);

    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const IO* f = static_cast<const IO*>(a.f);
    const IO* b = static_cast<const IO*>(a.b);
    const IO* g = static_cast<const IO*>(a.g);
    IO* cs = static_cast<IO*>(a.conv_state);

    for (int c = tid; c < 3 * D; c += REC_THREADS) {
        const int ch = conv_channel<D>(c, h, H);
        for (int j = 0; j < K; ++j) sm.cw[c][j] = a.conv_w[(size_t)ch * K + j];
        for (int r = 0; r < K - 1; ++r)
            sm.win[ring(r - (K - 1))][c] = ldv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch);
    }
    for (int i = tid; i < D; i += REC_THREADS) sm.dtb[i] = a.dt_bias[(size_t)h * D + i];
    const float ea = expf(a.A_log[h]);
    __syncthreads();

    for (int t = 0; t < L; ++t) {
        const size_t row = (size_t)row0 + t;
        const size_t rh = row * H + h;
        const int cur = ring(t);
        for (int c = tid; c < 3 * D; c += REC_THREADS) {
            float x;
            if (c < D) x = ldv(q + rh * D + c);
            else if (c < 2 * D) x = ldv(k + rh * D + (c - D));
            else x = ldv(v + rh * D + (c - 2 * D));
            sm.win[cur][c] = x;
        }
        for (int i = tid; i < D; i += REC_THREADS) sm.fr[i] = ldv(f + rh * D + i);
        __syncthreads();

        // conv window + SiLU, and the decay of each key dim
        for (int c = tid; c < 3 * D; c += REC_THREADS) {
            float acc = 0.0f;
            for (int j = 0; j < K; ++j) acc = __fmaf_rn(sm.cw[c][j], sm.win[ring(t - K + 1 + j)][c], acc);
            sm.act[c] = siluf_(acc);
        }
        for (int i = tid; i < D; i += REC_THREADS)
            sm.alpha[i] = __expf(log_alpha(a.gate_mode, a.lb, ea, sm.fr[i], sm.dtb[i]));
        __syncthreads();

        // q / k L2 norms and beta
        if (warp < 2) {
            float ss = 0.0f;
            for (int c = lane; c < D; c += 32) ss = __fmaf_rn(sm.act[warp * D + c], sm.act[warp * D + c], ss);
            ss = warp_sum(ss);
            if (lane == 0) sm.scal[warp] = rsqrtf(ss + a.l2_eps);
        } else if (warp == 2 && lane == 0) {
            sm.scal[2] = sigmoidf_(ldv(b + rh));
        }
        __syncthreads();
        for (int c = tid; c < D; c += REC_THREADS) {
            sm.qn[c] = sm.act[c] * sm.scal[0];
            sm.kn[c] = sm.act[D + c] * sm.scal[1];
        }
        __syncthreads();

        // S' = Diag(alpha) S ; kv = S'^T k (partial over this warp's rows)
        const float beta = sm.scal[2];
        float part[CPT];
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) part[cc] = 0.0f;
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const float ai = sm.alpha[r0 + rr], ki = sm.kn[r0 + rr];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                s[rr][cc] = __fmul_rn(ai, s[rr][cc]);
                part[cc] = __fmaf_rn(s[rr][cc], ki, part[cc]);
            }
        }
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) sm.red[warp][c0 + cc] = part[cc];
        __syncthreads();
        if (tid < D) {
            float kv = 0.0f;
#pragma unroll
            for (int w = 0; w < REC_WARPS; ++w) kv += sm.red[w][tid];
            sm.u[tid] = beta * (sm.act[2 * D + tid] - kv);
        }
        __syncthreads();

        // S = S' + k u^T ; o = S^T q (partial)
        float uc[CPT];
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) { uc[cc] = sm.u[c0 + cc]; part[cc] = 0.0f; }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const float ki = sm.kn[r0 + rr], qi = sm.qn[r0 + rr];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                s[rr][cc] = __fmaf_rn(ki, uc[cc], s[rr][cc]);
                part[cc] = __fmaf_rn(s[rr][cc], qi, part[cc]);
            }
        }
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) sm.red[warp][c0 + cc] = part[cc];
        __syncthreads();

        float o = 0.0f;
        if (tid < D) {
#pragma unroll
            for (int w = 0; w < REC_WARPS; ++w) o += sm.red[w][tid];
            o *= a.scale;
        }
        if (g != nullptr) {
            // sigmoid-gated RMSNorm over the head's D outputs
            float sq = tid < D ? o * o : 0.0f;
            sq = warp_sum(sq);
            if (lane == 0 && warp < D / 32) sm.scal[4 + warp] = sq;
            __syncthreads();
            if (tid < D) {
                float tot = 0.0f;
                for (int w = 0; w < D / 32; ++w) tot += sm.scal[4 + w];
                const float r = rsqrtf(tot * (1.0f / D) + a.norm_eps);
                const float w = a.norm_w ? a.norm_w[tid] : 1.0f;
                o = o * r * w * sigmoidf_(ldv(g + rh * D + tid));
            }
        }
        if (tid < D) store_out(a.out, rh * D + tid, o, a.out_bf16);

        if (MODE == REC_VERIFY) {
            float* lg = a.log_f + (((size_t)seq * a.W + t) * H + h) * (3 * D);
            if (tid < D) {
                lg[tid] = sm.alpha[tid];
                lg[D + tid] = sm.kn[tid];
                lg[2 * D + tid] = sm.u[tid];
            }
            IO* lr = static_cast<IO*>(a.log_raw) + ((size_t)seq * a.W + t) * conv_dim;
            for (int c = tid; c < 3 * D; c += REC_THREADS) stv(lr + conv_channel<D>(c, h, H), sm.win[cur][c]);
        }
        __syncthreads();
    }

    if (MODE != REC_VERIFY) {
        store_tile<D>(Sg, r0, c0, s);
        // new conv state: the last K-1 raw rows (older ones from the old state)
        for (int c = tid; c < 3 * D; c += REC_THREADS) {
            const int ch = conv_channel<D>(c, h, H);
            for (int r = 0; r < K - 1; ++r)
                stv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch, sm.win[ring(L - (K - 1) + r)][c]);
        }
    }
}

template <int D, typename IO>
__global__ void __launch_bounds__(REC_THREADS, 2) kda_commit_kernel(const CommitArgs a)
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, K = a.K, W = a.W;
    const int seq = blockIdx.x / H, h = blockIdx.x % H;
    const int conv_dim = H * 3 * D;
    const int slot = a.slots ? a.slots[seq] : seq;
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    const int acc = a.accepted[seq];
    if (acc < 0 || acc > W) {
        if (tid == 0 && h == 0) flag_status(a.dev_status, KDA_DEV_BAD_ACCEPTED);
        return;
    }
    if (acc == 0) return;

    float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
    const int r0 = warp * RPW, c0 = lane * CPT;
    float s[RPW][CPT];
    load_tile<D>(Sg, r0, c0, s);
    for (int t = 0; t < acc; ++t) {
        const float* lg = a.log_f + (((size_t)seq * W + t) * H + h) * (3 * D);
        float uc[CPT];
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) uc[cc] = lg[2 * D + c0 + cc];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const float ai = lg[r0 + rr], ki = lg[D + r0 + rr];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) s[rr][cc] = __fmaf_rn(ki, uc[cc], __fmul_rn(ai, s[rr][cc]));
        }
    }
    store_tile<D>(Sg, r0, c0, s);

    IO* cs = static_cast<IO*>(a.conv_state);
    const IO* raw = static_cast<const IO*>(a.log_raw);
    for (int c = tid; c < 3 * D; c += REC_THREADS) {
        const int ch = conv_channel<D>(c, h, H);
        float old[3], nw[3];
        for (int r = 0; r < K - 1; ++r) old[r] = ldv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch);
        for (int r = 0; r < K - 1; ++r) {
            const int src = acc - (K - 1) + r;  // window row, or < 0: old state row src + K - 1
            nw[r] = src >= 0 ? ldv(raw + ((size_t)seq * W + src) * conv_dim + ch) : old[src + K - 1];
        }
        for (int r = 0; r < K - 1; ++r) stv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch, nw[r]);
    }
}

template <int D, typename IO>
static cudaError_t launch_rec_d(int mode, const RecArgs& a, int units, cudaStream_t st)
{
    dim3 grid(units), block(REC_THREADS);
    if (mode == REC_PREFILL) kda_recurrent_kernel<D, IO, REC_PREFILL><<<grid, block, 0, st>>>(a);
    else if (mode == REC_DECODE) kda_recurrent_kernel<D, IO, REC_DECODE><<<grid, block, 0, st>>>(a);
    else kda_recurrent_kernel<D, IO, REC_VERIFY><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_recurrent(int mode, int io_bf16, const RecArgs& a, int units, cudaStream_t st)
{
    if (units <= 0) return cudaSuccess;
    switch (a.D) {
    case 32: return io_bf16 ? launch_rec_d<32, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<32, float>(mode, a, units, st);
    case 64: return io_bf16 ? launch_rec_d<64, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<64, float>(mode, a, units, st);
    case 128: return io_bf16 ? launch_rec_d<128, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<128, float>(mode, a, units, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_commit(int io_bf16, const CommitArgs& a, cudaStream_t st)
{
    const int units = a.B * a.H;
    if (units <= 0) return cudaSuccess;
    dim3 grid(units), block(REC_THREADS);
    switch (a.D) {
    case 32: if (io_bf16) kda_commit_kernel<32, __nv_bfloat16><<<grid, block, 0, st>>>(a); else kda_commit_kernel<32, float><<<grid, block, 0, st>>>(a); break;
    case 64: if (io_bf16) kda_commit_kernel<64, __nv_bfloat16><<<grid, block, 0, st>>>(a); else kda_commit_kernel<64, float><<<grid, block, 0, st>>>(a); break;
    case 128: if (io_bf16) kda_commit_kernel<128, __nv_bfloat16><<<grid, block, 0, st>>>(a); else kda_commit_kernel<128, float><<<grid, block, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kda
