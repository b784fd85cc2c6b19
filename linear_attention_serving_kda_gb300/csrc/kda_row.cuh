// kda_row.cuh -- one row of the KDA layer as the row-recurrent kernels run it
// (decode, verify windows, commit replay, the serial prefill).
//
// A (sequence, head) unit is processed by 256 threads.  The fp32 dk x dv
// state lives in registers while the unit's rows run, one tile of RPW key
// dims x CPT value dims per thread: in the register kernel warp w holds key
// dims [w*D/8, (w+1)*D/8) and lane l value dims [l*D/32, (l+1)*D/32), so each
// warp touches whole D-float rows (coalesced, vector accesses) and the two
// key-dim reductions per row (S'^T k and S^T q) are an in-register chain over
// the tile's key dims followed by a fixed-order sum over the key-dim blocks.
//
// Every row is formed by the expressions of row_conv, row_delta and row_out,
// in their order -- S' = alpha * S (rounded), then S = fma(k, u, S') -- on the
// same tiles with the same reduction trees.  So a verified row has the bits of
// a decoded row, and a committed state the bits of serial decode (TensorFold
// issue #850, Oct 15 comment: a window logs each row's decay, normalized key
// and update, and replaying them gives the bits of rows decoded one at a time;
// Oct 19 comment: preserve rounding, reduction order, replay).
#pragma once

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {

constexpr int REC_THREADS = 256;
constexpr int REC_WARPS = REC_THREADS / 32;

template <int D> struct RecShape {
    static constexpr int CPT = D / 32;        // state columns per lane
    static constexpr int RPW = D / REC_WARPS; // state rows per warp
};

template <int D> struct RowSmem {
    float win[4][3 * D];      // ring of the last 4 raw conv rows (this head's q|k|v channels)
    float cw[3 * D][4];       // conv taps
    float dtb[D];             // dt_bias of this head
    float act[3 * D];         // post-SiLU q', k', v'
    float alpha[D], fr[D];
    float red[REC_WARPS][D];  // cross-warp partial sums of S'^T k
    float red2[REC_WARPS][D]; // cross-warp partial sums of S^T q
    float nrm[8];             // per-warp sums of squares: q' [0, D/32), k' [D/32, 2D/32)
    float scal[8];
};

struct RowConst {
    int gate_mode;
    float lb, ea, l2_eps, norm_eps, scale;
    const float* norm_w;
};

__device__ __forceinline__ int ring(int x) { return x & 3; }

// Barrier over the 256 row threads only (a streaming CTA also has a producer warp).
__device__ __forceinline__ void row_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Global channel of local channel c (q | k | v of head h) in the conv layout.
template <int D> __device__ __forceinline__ int conv_channel(int c, int h, int H)
{
    if (c < D) return h * D + c;
    if (c < 2 * D) return H * D + h * D + (c - D);
    return 2 * H * D + h * D + (c - 2 * D);
}

template <int D, typename Src>
__device__ __forceinline__ void load_tile(const Src* Sg, int r0, int c0,
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

template <int D>
__device__ __forceinline__ void load_tile_smem(const float* Ss, int r0, int c0,
                                               float (&s)[RecShape<D>::RPW][RecShape<D>::CPT])
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    static_assert(CPT == 4, "shared-memory tile path is for D = 128");
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        float4 x = *reinterpret_cast<const float4*>(Ss + (r0 + rr) * D + c0);
        s[rr][0] = x.x; s[rr][1] = x.y; s[rr][2] = x.z; s[rr][3] = x.w;
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

// One row of the layer for one (sequence, head); called by all 256 threads,
// in two steps.
//
// row_conv: on entry sm.cw / sm.dtb hold the head's parameters; win(c, j) is
// raw value j (oldest first, j = K-1 the current row) of local channel c
// (q | k | v), fr(i) the gate of key dim i.  Leaves the post-SiLU q|k|v row in
// sm.act, each key dim's decay in sm.alpha and per-warp sums of squares of q'
// and k' in sm.nrm.  The 3D conv channels and the D decays are 4D items taken
// round-robin by the threads (two each at D = 128); the q and k channels fill
// whole warps of the first round.  The thread that takes item c < 3D must be
// the one that loaded sm.cw[c] (item 3D + i: sm.dtb[i]) when the caller
// relies on that instead of a barrier.
//
// row_delta: the q and k inverse norms and beta into sm.scal[0..2], the delta
// rule on S (in registers: warp w owns rows [RPW w, +RPW), lane l columns
// [CPT l, +CPT)), sm.red the per-warp partials of S'^T k (so the normalised key
// is act[D + i] * scal[1] and the update u_j = beta (act[2D + j] - sum_w
// red[w][j]), the same expressions as here), and sm.red2 the per-warp partials
// of S^T q.  No barrier after the last step: the caller may store S first.
//
// row_out: the output of column tid (tid < D), with the optional
// sigmoid-gated RMSNorm; gval is the output gate of column tid.
//
// Every warp forms the norms, beta and the update of its own columns itself
// from the same shared values in the same order (identical bits everywhere).
// Decode, verify and commit use these functions and the expressions they log,
// so a verified row has the bits of a decoded one.
template <int D, typename Win, typename Fr>
__device__ __forceinline__ void row_conv(RowSmem<D>& sm, int K, const RowConst& rc, Win win, Fr fr)
{
    const int tid = threadIdx.x, lane = tid & 31;
    for (int it = tid; it < 4 * D; it += REC_THREADS) {
        if (it < 3 * D) {
            float acc = 0.0f;
            for (int j = 0; j < K; ++j) acc = __fmaf_rn(sm.cw[it][j], win(it, j), acc);
            const float x = siluf_(acc);
            sm.act[it] = x;
            if (it < 2 * D) {  // warp-uniform: D is a multiple of 32
                const float ss = warp_sum(x * x);
                if (lane == 0) sm.nrm[it >> 5] = ss;
            }
        } else {
            const int i = it - 3 * D;
            sm.alpha[i] = exp_sfu(log_alpha(rc.gate_mode, rc.lb, rc.ea, fr(i), sm.dtb[i]));
        }
    }
    row_sync();
}

template <int D>
__device__ __forceinline__ void row_delta(RowSmem<D>& sm, float (&s)[RecShape<D>::RPW][RecShape<D>::CPT],
                                          const RowConst& rc, float bval)
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT, NP = D / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = warp * RPW, c0 = lane * CPT;

    float sq = 0.0f, sk = 0.0f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        sq += sm.nrm[p];
        sk += sm.nrm[NP + p];
    }
    const float rq = rsqrtf(sq + rc.l2_eps);
    const float rk = rsqrtf(sk + rc.l2_eps);
    const float beta = sigmoidf_(bval);
    if (tid == 0) {
        sm.scal[0] = rq;
        sm.scal[1] = rk;
        sm.scal[2] = beta;
    }

    // S' = Diag(alpha) S ; kv = S'^T k (partial over this warp's rows).  Column
    // pairs in packed f32x2 arithmetic: the same rounded operations per element.
    float kr[RPW], part[CPT];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) kr[rr] = sm.act[D + r0 + rr] * rk;
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) part[cc] = 0.0f;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const float ai = sm.alpha[r0 + rr];
        if constexpr (CPT % 2 == 0) {
#pragma unroll
            for (int cc = 0; cc < CPT; cc += 2) {
                const float2 sp = __fmul2_rn(make_float2(ai, ai), make_float2(s[rr][cc], s[rr][cc + 1]));
                const float2 pp = __ffma2_rn(sp, make_float2(kr[rr], kr[rr]), make_float2(part[cc], part[cc + 1]));
                s[rr][cc] = sp.x;
                s[rr][cc + 1] = sp.y;
                part[cc] = pp.x;
                part[cc + 1] = pp.y;
            }
        } else {
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                s[rr][cc] = __fmul_rn(ai, s[rr][cc]);
                part[cc] = __fmaf_rn(s[rr][cc], kr[rr], part[cc]);
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) sm.red[warp][c0 + cc] = part[cc];
    row_sync();

    // u of this thread's columns: the partials summed in warp order
    float uc[CPT], kv[CPT];
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) kv[cc] = 0.0f;
#pragma unroll
    for (int w = 0; w < REC_WARPS; ++w) {
        if constexpr (CPT == 4) {
            const float4 r4 = *reinterpret_cast<const float4*>(&sm.red[w][c0]);
            kv[0] += r4.x;
            kv[1] += r4.y;
            kv[2] += r4.z;
            kv[3] += r4.w;
        } else {
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) kv[cc] += sm.red[w][c0 + cc];
        }
    }
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
        uc[cc] = beta * (sm.act[2 * D + c0 + cc] - kv[cc]);
        part[cc] = 0.0f;
    }

    // S = S' + k u^T ; o = S^T q (partial)
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const float qi = sm.act[r0 + rr] * rq;
        if constexpr (CPT % 2 == 0) {
#pragma unroll
            for (int cc = 0; cc < CPT; cc += 2) {
                const float2 sn = __ffma2_rn(make_float2(kr[rr], kr[rr]), make_float2(uc[cc], uc[cc + 1]),
                                             make_float2(s[rr][cc], s[rr][cc + 1]));
                const float2 pp = __ffma2_rn(sn, make_float2(qi, qi), make_float2(part[cc], part[cc + 1]));
                s[rr][cc] = sn.x;
                s[rr][cc + 1] = sn.y;
                part[cc] = pp.x;
                part[cc + 1] = pp.y;
            }
        } else {
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                s[rr][cc] = __fmaf_rn(kr[rr], uc[cc], s[rr][cc]);
                part[cc] = __fmaf_rn(s[rr][cc], qi, part[cc]);
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) sm.red2[warp][c0 + cc] = part[cc];
}

template <int D>
__device__ __forceinline__ float row_out(RowSmem<D>& sm, const RowConst& rc, float gval, bool has_g)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    row_sync();
    float o = 0.0f;
    if (tid < D) {
#pragma unroll
        for (int w = 0; w < REC_WARPS; ++w) o += sm.red2[w][tid];
        o *= rc.scale;
    }
    if (has_g) {
        // sigmoid-gated RMSNorm over the head's D outputs
        float sq = tid < D ? o * o : 0.0f;
        sq = warp_sum(sq);
        if (lane == 0 && warp < D / 32) sm.scal[4 + warp] = sq;
        row_sync();
        if (tid < D) {
            float tot = 0.0f;
            for (int w = 0; w < D / 32; ++w) tot += sm.scal[4 + w];
            const float r = rsqrtf(tot * (1.0f / D) + rc.norm_eps);
            const float w = rc.norm_w ? rc.norm_w[tid] : 1.0f;
            o = o * r * w * sigmoidf_(gval);
        }
    }
    return o;
}

// conv, delta rule and output of a row whose raw values sit in the window ring
template <int D>
__device__ __forceinline__ float row_step(RowSmem<D>& sm, float (&s)[RecShape<D>::RPW][RecShape<D>::CPT],
                                          int t, int K, const RowConst& rc, float bval, float gval, bool has_g)
{
    row_conv<D>(sm, K, rc, [&](int c, int j) { return sm.win[ring(t - K + 1 + j)][c]; },
                [&](int i) { return sm.fr[i]; });
    row_delta<D>(sm, s, rc, bval);
    return row_out<D>(sm, rc, gval, has_g);
}

// The update u_j of the last row_step (column j), from what it left in shared memory.
template <int D> __device__ __forceinline__ float row_update(const RowSmem<D>& sm, int j)
{
    float kv = 0.0f;
#pragma unroll
    for (int w = 0; w < REC_WARPS; ++w) kv += sm.red[w][j];
    return sm.scal[2] * (sm.act[2 * D + j] - kv);
}

// streaming kernels (decode, commit) at dk = dv = 128: 8 row warps + a producer warp
constexpr int DEC_D = 128;
constexpr int DEC_THREADS = REC_THREADS + 32;

// SM count of the current device, remembered per device (an atomic: several
// host threads may ask at once; each stores the same value)
static inline int sm_count()
{
    static std::atomic<int> n[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int c = n[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
        c = c > 0 ? c : 148;
        n[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

}  // namespace kda
