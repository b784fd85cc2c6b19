// kda_scan.cu -- chunk-parallel prefill of long sequences by an affine state
// scan (the context-parallel form of the chunked prefill).
//
// The delta rule is linear in the state: over any run of rows the state at
// the end is S_out = M S_in + N, and every output row is o_r = obar_r +
// psi_r S_in, where (N, obar) are what the rows give from a zero state and
// (M, psi) what they give from the identity with the values v set to zero
// (then u = -beta S'^T k, so the recurrence carries S_in alone).  So each
// sequence is cut into P segments of whole 64-row chunks (TensorFold issue
// #850, Oct 15 comment: a segment's rows run in chunks from its first row),
// and
//   1. every segment runs from a zero state (its end state N_p and raw
//      outputs obar) and every segment but the first also from the identity
//      with zero values (its transfer M_p and output corrections psi) -- both
//      as units of one launch of the fused chunk kernel;
//   2. a scan per (sequence, head) walks the segments: S_1 is the first
//      segment's end state and S_{p+1} = M_p S_p + N_p;
//   3. a fix-up adds psi_r S_p to every output row of segment p >= 1 and
//      applies the sigmoid-gated RMSNorm.
// Segments are independent, so on several GPUs each takes its own (steps 1
// and 3) and only the scan's states travel between them; here they share one
// GPU.  The results agree with the serial recurrence to rounding, not bit for
// bit with kda_prefill_varlen (other summation order).
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace scn {

constexpr int D = 128;
constexpr int C = 64;

// Segment plan (one block).  Sequence s of L rows is cut into P segments of
// seg = round_up(ceil(L / P), 64) rows (the last ones may be short or
// empty).  pseudo-sequence j = s P + p covers rows [pcu[j], pcu[j + 1]).
// Unit slots of the chunk kernel: zero-state run j -> j, transfer run
// (p >= 1) -> NP + j, -1 when the sequence is skipped (negative slot, bad
// slot or bad cu_seqlens).  tiles[j]: 64-row output tiles before
// pseudo-sequence j.
__global__ void kda_scan_plan_kernel(const int32_t* cu, const int32_t* slots, int N, int T, int P, int num_slots,
                                     int32_t* pcu, int32_t* pslots, int32_t* tiles, int32_t* dev_status)
{
    const int NP = N * P;
    for (int s = threadIdx.x; s < N; s += blockDim.x) {
        const int c0 = cu[s], c1 = cu[s + 1];
        const bool ok_cu = c0 >= 0 && c1 >= c0 && c1 <= T;
        const int sl = slots ? slots[s] : s;
        if (!ok_cu) flag_status(dev_status, KDA_DEV_BAD_SEQLENS);
        else if (sl >= num_slots) flag_status(dev_status, KDA_DEV_BAD_SLOT);
        const bool run = ok_cu && sl >= 0 && sl < num_slots;
        const int L = ok_cu ? c1 - c0 : 0;
        const int per = (L + P - 1) / P;
        const int seg = (per + C - 1) / C * C;
        for (int p = 0; p < P; ++p) {
            const int j = s * P + p;
            // an invalid sequence keeps pcu monotone with empty segments at c0 (clamped)
            const int base = ok_cu ? c0 : min(max(c0, 0), T);
            pcu[j] = base + min(p * seg, L);
            pslots[j] = run ? j : -1;
            pslots[NP + j] = (run && p > 0) ? NP + j : -1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // segments of consecutive sequences are contiguous: segment j ends where j + 1 starts
        pcu[NP] = min(max(cu[N], 0), T);
        int t = 0;
        for (int j = 0; j < NP; ++j) {
            tiles[j] = t;
            t += (max(pcu[j + 1] - pcu[j], 0) + C - 1) / C;
        }
        tiles[NP] = t;
    }
}

// The end row of pseudo-sequence j.
__device__ __forceinline__ int seg_end(const int32_t* pcu, int j) { return pcu[j + 1]; }

// Initial states of every unit of the chunk-kernel launch (one block per
// (pseudo-sequence, head) of each run): recurrent state -- the sequence's own
// for its first segment, zero for the other zero-state runs, the identity for
// transfer runs -- and conv state -- the sequence's own for its first segment,
// else the K-1 raw rows before the segment (from the carried conv state where
// they fall before the sequence).
template <typename IO>
__global__ void kda_scan_init_kernel(const int32_t* cu, const int32_t* slots, int N, int P, int H, int K,
                                     const int32_t* pcu, const int32_t* pslots, const IO* q, const IO* k,
                                     const IO* v, const IO* conv_state, const float* rec_state, IO* wconv,
                                     float* wrec)
{
    const int NP = N * P;
    const int unit = blockIdx.x;  // run * NP + j
    const int h = blockIdx.y;
    const int j = unit % NP, run = unit / NP;
    const int s = j / P, p = j % P;
    if (pslots[unit] < 0) return;
    const int sl = slots ? slots[s] : s;
    // recurrent state
    float* dst = wrec + ((size_t)unit * H + h) * D * D;
    const float* src = rec_state + ((size_t)sl * H + h) * D * D;
    for (int e = threadIdx.x * 4; e < D * D; e += blockDim.x * 4) {
        float4 x;
        if (run == 0 && p == 0) {
            x = *reinterpret_cast<const float4*>(src + e);
        } else if (run == 0) {
            x = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int i = e / D, c = e % D;  // identity: 1 where column == row
            x = make_float4(c == i ? 1.f : 0.f, c + 1 == i ? 1.f : 0.f, c + 2 == i ? 1.f : 0.f, c + 3 == i ? 1.f : 0.f);
        }
        *reinterpret_cast<float4*>(dst + e) = x;
    }
    // conv state: this head's q, k, v channels of the K-1 rows
    const int conv_dim = 3 * H * D;
    const int c0 = cu[s], start = pcu[j];
    for (int e = threadIdx.x; e < (K - 1) * 3 * D; e += blockDim.x) {
        const int r = e / (3 * D), ch = e % (3 * D), tsel = ch / D, cc = ch % D;
        const size_t col = (size_t)tsel * H * D + (size_t)h * D + cc;
        IO val;
        const int x = start - (K - 1) + r;  // absolute row
        if (p == 0 || x < c0) {
            // from the carried conv state: its row K-1 + (x - c0) (for p == 0, row r)
            const int cr = p == 0 ? r : (K - 1) + (x - c0);
            val = conv_state[((size_t)sl * (K - 1) + cr) * conv_dim + col];
        } else {
            const IO* base = tsel == 0 ? q : (tsel == 1 ? k : v);
            val = base[((size_t)x * H + h) * D + cc];
        }
        wconv[((size_t)unit * (K - 1) + r) * conv_dim + col] = val;
    }
}

// The scan (one block per (sequence, head)): S = the first segment's end
// state; for p = 1 .. P-1: keep S as segment p's start state (into the
// zero-state run's slot, whose N_p is read first) and S <- M_p S + N_p; the
// last S is the sequence's final state, and the last segment's conv state
// (the sequence's last K-1 raw rows) its final conv state.
template <typename IO>
__global__ void __launch_bounds__(256, 1)
    kda_scan_states_kernel(const int32_t* slots, int N, int P, int H, int K, const int32_t* pslots, float* wrec,
                           const IO* wconv, float* rec_state, IO* conv_state)
{
    extern __shared__ __align__(16) float scn_smem[];
    float* S = scn_smem;          // [D][D]
    float* M = scn_smem + D * D;  // [D][D]
    const int NP = N * P;
    const int s = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (pslots[s * P] < 0) return;  // skipped sequence
    const int sl = slots ? slots[s] : s;
    // thread tile: rows [8 (tid / 16), +8), columns [8 (tid % 16), +8)
    const int i0 = 8 * (tid >> 4), j0 = 8 * (tid & 15);
    auto rec = [&](int unit) { return wrec + ((size_t)unit * H + h) * D * D; };
    for (int e = tid * 4; e < D * D; e += 256 * 4)
        *reinterpret_cast<float4*>(S + e) = *reinterpret_cast<const float4*>(rec(s * P) + e);
    for (int p = 1; p < P; ++p) {
        const int ja = s * P + p, jb = NP + ja;
        for (int e = tid * 4; e < D * D; e += 256 * 4)
            *reinterpret_cast<float4*>(M + e) = *reinterpret_cast<const float4*>(rec(jb) + e);
        float acc[8][8];
        const float* Nn = rec(ja);
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int b = 0; b < 8; b += 4) {
                const float4 x = *reinterpret_cast<const float4*>(Nn + (size_t)(i0 + a) * D + j0 + b);
                acc[a][b] = x.x; acc[a][b + 1] = x.y; acc[a][b + 2] = x.z; acc[a][b + 3] = x.w;
            }
        __syncthreads();  // M staged; every thread has read its part of N_p
        for (int kk = 0; kk < D; ++kk) {
            float mv[8], sv[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) mv[a] = M[(i0 + a) * D + kk];
            const float4 s0 = *reinterpret_cast<const float4*>(S + kk * D + j0);
            const float4 s1 = *reinterpret_cast<const float4*>(S + kk * D + j0 + 4);
            sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w;
            sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = __fmaf_rn(mv[a], sv[b], acc[a][b]);
        }
        // segment p's start state into the zero-state slot (its N_p has been read)
        float* St = rec(ja);
        for (int e = tid * 4; e < D * D; e += 256 * 4)
            *reinterpret_cast<float4*>(St + e) = *reinterpret_cast<const float4*>(S + e);
        __syncthreads();  // S read by every thread
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int b = 0; b < 8; b += 4)
                *reinterpret_cast<float4*>(S + (i0 + a) * D + j0 + b) =
                    make_float4(acc[a][b], acc[a][b + 1], acc[a][b + 2], acc[a][b + 3]);
        __syncthreads();
    }
    float* out = rec_state + ((size_t)sl * H + h) * D * D;
    for (int e = tid * 4; e < D * D; e += 256 * 4)
        *reinterpret_cast<float4*>(out + e) = *reinterpret_cast<const float4*>(S + e);
    // final conv state: the last segment's (the sequence's last K-1 raw rows), this head's channels
    const int conv_dim = 3 * H * D, last = s * P + P - 1;
    for (int e = tid; e < (K - 1) * 3 * D; e += 256) {
        const int r = e / (3 * D), ch = e % (3 * D), tsel = ch / D, cc = ch % D;
        const size_t col = (size_t)tsel * H * D + (size_t)h * D + cc;
        conv_state[((size_t)sl * (K - 1) + r) * conv_dim + col] = wconv[((size_t)last * (K - 1) + r) * conv_dim + col];
    }
}

// The fix-up: o = obar (+ psi S_p for segments p >= 1), then the optional
// sigmoid-gated RMSNorm, stored in the output type.  Grid (tiles, H): one
// CTA per 64-row output tile and head (any CTA past the last tile returns).
// Thread (row group
// gq = tid / 32, lane) owns rows [8 gq, +8) and columns [4 lane, +4); each
// output sums obar and the 128 terms psi_ri S_ij in key order i.  The psi
// tile is stored transposed (key dim major) with its 8-row groups permuted by
// the key dim (an XOR of the row index's upper bits), so the 8 rows a thread
// needs for one key dim are 32 contiguous bytes and the transposing stores
// spread over the banks.
constexpr int FX_PT = 68;  // row pitch (floats) of the transposed psi tile

__device__ __forceinline__ int fx_row(int r, int i) { return r ^ (8 * ((i >> 2) & 7)); }

__global__ void __launch_bounds__(256, 2)
    kda_scan_fixup_kernel(int N, int P, int H, const int32_t* pcu, const int32_t* pslots, const int32_t* tiles,
                          const float* obar, const float* psi, const float* wrec, const void* g, const float* norm_w,
                          float norm_eps, int has_g, void* out, int out_bf16)
{
    extern __shared__ __align__(16) float scn_smem[];
    float* Ss = scn_smem;          // [D][D] segment start state
    float* Pt = scn_smem + D * D;  // [D][FX_PT] psi tile, transposed and row-permuted
    const int NP = N * P;
    const int h = blockIdx.y, tid = threadIdx.x;
    const int ntiles = tiles[NP];
    const int gq = tid >> 5, lane = tid & 31, c0 = 4 * lane;
    int loaded = -1;  // pseudo-sequence whose start state is in Ss
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        int lo = 0, hi = NP - 1;  // the pseudo-sequence j with tiles[j] <= t < tiles[j + 1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tiles[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const int j = lo, p = j % P;
        if (pslots[j] < 0) continue;  // block-uniform
        const int r0 = pcu[j] + (t - tiles[j]) * C;
        const int nrows = min(C, seg_end(pcu, j) - r0);
        if (nrows <= 0) continue;
        float2 acc[4][4];  // (rows 8 gq + 2 a, + 1) x column c0 + b
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
            const int ra = 8 * gq + 2 * a;
            if (ra < nrows) x0 = *reinterpret_cast<const float4*>(obar + ((size_t)(r0 + ra) * H + h) * D + c0);
            if (ra + 1 < nrows) x1 = *reinterpret_cast<const float4*>(obar + ((size_t)(r0 + ra + 1) * H + h) * D + c0);
            acc[a][0] = make_float2(x0.x, x1.x);
            acc[a][1] = make_float2(x0.y, x1.y);
            acc[a][2] = make_float2(x0.z, x1.z);
            acc[a][3] = make_float2(x0.w, x1.w);
        }
        if (p > 0) {
            __syncthreads();  // the previous tile's reads of Ss and Pt are done
            if (loaded != j) {
                const float* St = wrec + ((size_t)j * H + h) * D * D;  // segment p's start state
                for (int e = tid * 4; e < D * D; e += 256 * 4)
                    *reinterpret_cast<float4*>(Ss + e) = *reinterpret_cast<const float4*>(St + e);
                loaded = j;
            }
            for (int e = tid * 4; e < C * D; e += 256 * 4) {
                const int r = e / D, i = e % D;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < nrows) x = *reinterpret_cast<const float4*>(psi + ((size_t)(r0 + r) * H + h) * D + i);
                const int rr = fx_row(r, i);  // i .. i + 3 share (i >> 2)
                Pt[(i + 0) * FX_PT + rr] = x.x;
                Pt[(i + 1) * FX_PT + rr] = x.y;
                Pt[(i + 2) * FX_PT + rr] = x.z;
                Pt[(i + 3) * FX_PT + rr] = x.w;
            }
            __syncthreads();
#pragma unroll 4
            for (int i = 0; i < D; ++i) {
                const float* pc = Pt + i * FX_PT + fx_row(8 * gq, i);  // rows 8 gq .. + 7 of key dim i
                const float4 p0 = *reinterpret_cast<const float4*>(pc);
                const float4 p1 = *reinterpret_cast<const float4*>(pc + 4);
                const float4 sv = *reinterpret_cast<const float4*>(Ss + i * D + c0);
                const float2 pr[4] = {make_float2(p0.x, p0.y), make_float2(p0.z, p0.w), make_float2(p1.x, p1.y),
                                      make_float2(p1.z, p1.w)};
                const float2 s2[4] = {make_float2(sv.x, sv.x), make_float2(sv.y, sv.y), make_float2(sv.z, sv.z),
                                      make_float2(sv.w, sv.w)};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = __ffma2_rn(pr[a], s2[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const int r = 8 * gq + a;
            float y[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) y[b] = (a & 1) ? acc[a >> 1][b].y : acc[a >> 1][b].x;
            if (has_g) {
                const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
                const float rn = rsqrtf(ss * (1.0f / D) + norm_eps);
                if (r < nrows) {
                    const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(g) + ((size_t)(r0 + r) * H + h) * D + c0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const float w = norm_w ? norm_w[c0 + b] : 1.0f;
                        y[b] = y[b] * rn * w * sigmoidf_(__bfloat162float(gb[b]));
                    }
                }
            }
            if (r < nrows) {
                const size_t o = ((size_t)(r0 + r) * H + h) * D + c0;
#pragma unroll
                for (int b = 0; b < 4; ++b) store_out(out, o + b, y[b], out_bf16);
            }
        }
    }
}

}  // namespace scn

// Workspace of kda_prefill_scan (1 KiB-aligned parts): pcu [NP + 1], unit
// slots [2 NP], tile offsets [NP + 1], the chunk kernel's schedule [2 NP],
// recurrent states [2 NP][H][128][128] fp32, conv states [2 NP][K-1][conv_dim]
// (io type), obar and psi [T][H][128] fp32 each.
struct ScanWs {
    size_t pcu, pslots, tiles, sched, wrec, wconv, obar, psi, total;
};

static size_t al1k(size_t x) { return (x + 1023) & ~size_t(1023); }

static ScanWs scan_layout(const kda_params* p, int N, int T, int P)
{
    ScanWs w;
    const size_t NP = (size_t)N * P, H = p->num_heads, conv_dim = 3 * H * scn::D;
    const size_t io = p->io_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    size_t o = 0;
    w.pcu = o; o += al1k((NP + 1) * 4);
    w.pslots = o; o += al1k(2 * NP * 4);
    w.tiles = o; o += al1k((NP + 1) * 4);
    w.sched = o; o += al1k(2 * NP * 4);
    w.wrec = o; o += al1k(2 * NP * H * scn::D * scn::D * 4);
    w.wconv = o; o += al1k(2 * NP * (size_t)(p->conv_kernel - 1) * conv_dim * io);
    w.obar = o; o += al1k((size_t)T * H * scn::D * 4);
    w.psi = o; o += al1k((size_t)T * H * scn::D * 4);
    w.total = o;
    return w;
}

size_t prefill_scan_workspace_bytes(const kda_params* p, int N, int T, int P)
{
    return scan_layout(p, N, T, P).total;
}

cudaError_t launch_prefill_scan(const kda_params* p, const ChunkArgs& a0, int P, unsigned char* ws, cudaStream_t st)
{
    using namespace scn;
    const int N = a0.N, T = a0.T, H = a0.H, K = a0.K, NP = N * P;
    const ScanWs w = scan_layout(p, N, T, P);
    int32_t* pcu = reinterpret_cast<int32_t*>(ws + w.pcu);
    int32_t* pslots = reinterpret_cast<int32_t*>(ws + w.pslots);
    int32_t* tiles = reinterpret_cast<int32_t*>(ws + w.tiles);
    float* wrec = reinterpret_cast<float*>(ws + w.wrec);
    __nv_bfloat16* wconv = reinterpret_cast<__nv_bfloat16*>(ws + w.wconv);
    float* obar = reinterpret_cast<float*>(ws + w.obar);
    float* psi = reinterpret_cast<float*>(ws + w.psi);

    kda_scan_plan_kernel<<<1, 256, 0, st>>>(a0.cu_seqlens, a0.slots, N, T, P, a0.num_slots, pcu, pslots, tiles,
                                            a0.dev_status);
    kda_scan_init_kernel<__nv_bfloat16><<<dim3(2 * NP, H), 256, 0, st>>>(
        a0.cu_seqlens, a0.slots, N, P, H, K, pcu, pslots, static_cast<const __nv_bfloat16*>(a0.q),
        static_cast<const __nv_bfloat16*>(a0.k), static_cast<const __nv_bfloat16*>(a0.v),
        static_cast<const __nv_bfloat16*>(a0.conv_state), a0.rec_state, wconv, wrec);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // both runs of every segment in one launch of the fused chunk kernel
    ChunkArgs c = a0;
    c.N = 2 * NP;
    c.num_slots = 2 * NP;
    c.cu_seqlens = pcu;
    c.slots = pslots;
    c.conv_state = wconv;
    c.rec_state = wrec;
    c.out = obar;
    c.out2 = psi;
    c.out_bf16 = 0;
    c.g = nullptr;  // raw outputs: the norm comes after the fix-up
    c.nsplit = NP;
    c.schedule = reinterpret_cast<int32_t*>(ws + w.sched);
    c.split_ws = nullptr;
    c.dbg_chains_only_polls = 0;
    if ((e = launch_chunk(1, c, st)) != cudaSuccess) return e;

    static PerDeviceOnce attr;
    const int smem_scan = 2 * D * D * 4, smem_fix = (D * D + D * FX_PT) * 4;
    e = attr.run([&](int) {
        cudaError_t r = cudaFuncSetAttribute(kda_scan_states_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_scan);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(kda_scan_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_fix);
        return r;
    });
    if (e != cudaSuccess) return e;
    kda_scan_states_kernel<__nv_bfloat16><<<dim3(N, H), 256, smem_scan, st>>>(
        a0.slots, N, P, H, K, pslots, wrec, wconv, a0.rec_state, static_cast<__nv_bfloat16*>(a0.conv_state));
    // one CTA per (64-row tile, head): many tiles in flight hide the loads
    const int max_tiles = (T + C - 1) / C + NP;
    kda_scan_fixup_kernel<<<dim3(max_tiles, H), 256, smem_fix, st>>>(N, P, H, pcu, pslots, tiles, obar, psi, wrec,
                                                                    a0.g, a0.norm_w, a0.norm_eps, a0.g != nullptr,
                                                                    a0.out, a0.out_bf16);
    return cudaGetLastError();
}

}  // namespace kda
