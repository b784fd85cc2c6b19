// kda_recurrent.cu -- row-recurrent KDA kernels for sm_103a: verify windows
// (and commit fused into the next window), commit, and the row-by-row prefill
// for the shapes the chunk kernel does not take (fp32 rows, dk < 128).  Rows
// follow kda_row.cuh, so they carry decode's bits.  At dk = dv = 128 verify
// windows and that prefill regroup the thread tiles so that a row's sums stay
// inside a warp (kda_verify_warp_kernel) and commit streams through
// shared-memory stages like decode (kda_commit_stream_kernel); other widths
// run the register kernel, one CTA per unit.
#include "kda_row.cuh"

namespace kda {

// ------------------------------------------------------------------------
// Staged window rows.  A verify window's draft rows (q, k, v, gate f, output
// gate g) are copied into shared memory in blocks of VWB rows with 16-byte
// cp.async pieces, the next block while the current one runs, so no row of
// the window waits on a global load; a commit's log rows (alpha | k^ | u) are
// staged the same way before they are replayed.  The values are the ones the
// per-row global loads would read, so the arithmetic and its bits are
// unchanged.

constexpr int VWB = 8;  // window rows per staged block

template <int D, typename IO> struct VerBuf {
    IO rows[VWB][5][D];  // q, k, v, f, g of each row of the block
    float bv[VWB];       // beta logits
};

template <int D, typename IO> struct VerSmem {
    VerBuf<D, IO> buf[2];      // double-buffered blocks
    float plog[VWB][3 * D];    // a block of log rows to replay (commit)
};

// Issue the copies of window rows [t0, t0 + nr) of unit (seq, h) into vb (all
// threads; one commit group).  The beta logits are returned as raw values of
// the threads tid < nr, to be written into vb.bv when the block is published,
// so no thread waits on their load here.
template <int D, typename IO>
__device__ __forceinline__ IO stage_window_rows(VerBuf<D, IO>& vb, const RecArgs& a, int seq, int h, int t0, int nr)
{
    constexpr int EPP = 16 / (int)sizeof(IO);  // elements per 16-byte piece
    constexpr int PIECES = D / EPP;            // pieces per row
    const int ntens = a.g != nullptr ? 5 : 4;
    for (int idx = threadIdx.x; idx < nr * ntens * PIECES; idx += REC_THREADS) {
        const int piece = idx % PIECES, rest = idx / PIECES, tens = rest % ntens, r = rest / ntens;
        const size_t rh = ((size_t)seq * a.W + t0 + r) * a.H + h;
        const void* base = tens == 0 ? a.q : tens == 1 ? a.k : tens == 2 ? a.v : tens == 3 ? a.f : a.g;
        ptx::cp_async16(&vb.rows[r][tens][piece * EPP], static_cast<const IO*>(base) + rh * D + piece * EPP, 16);
    }
    ptx::cp_async_commit();
    const IO* b = static_cast<const IO*>(a.b);
    IO braw{};
    if (threadIdx.x < nr) braw = b[((size_t)seq * a.W + t0 + threadIdx.x) * a.H + h];
    return braw;
}

// Issue the copies of log rows [t0, t0 + nr) (alpha | k^ | u, fp32) of unit
// (seq, h) into plog (all threads; one commit group).
template <int D>
__device__ __forceinline__ void stage_log_rows(float (&plog)[VWB][3 * D], const float* log_f, int W, int H, int seq,
                                               int h, int t0, int nr)
{
    constexpr int PIECES = 3 * D / 4;
    for (int idx = threadIdx.x; idx < nr * PIECES; idx += REC_THREADS) {
        const int piece = idx % PIECES, r = idx / PIECES;
        ptx::cp_async16(&plog[r][piece * 4], log_f + (((size_t)seq * W + t0 + r) * H + h) * (3 * D) + piece * 4, 16);
    }
    ptx::cp_async_commit();
}

// Replay staged log rows [0, nr) onto this thread's part of the state:
// S <- fma(k^, u, alpha * S), the expression of the decoded row.
template <int D>
__device__ __forceinline__ void replay_log_rows(const float (&plog)[VWB][3 * D], int nr,
                                                float (&s)[RecShape<D>::RPW][RecShape<D>::CPT])
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = warp * RPW, c0 = lane * CPT;
    for (int t = 0; t < nr; ++t) {
        const float* lg = plog[t];
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
}

// ------------------------------------------------------------------------
// Register kernel: one CTA per unit, all of the unit's rows.

template <int D, typename IO, int MODE>
__global__ void __launch_bounds__(REC_THREADS, 2) kda_recurrent_kernel(const RecArgs a)
{
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    __shared__ RowSmem<D> sm;
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
    int acc = 0;  // REC_COMMIT_VERIFY: rows of the previous window to commit first
    if (MODE == REC_COMMIT_VERIFY) {
        acc = a.accepted[seq];
        if (acc < 0 || acc > a.W) {
            if (tid == 0 && h == 0) flag_status(a.dev_status, KDA_DEV_BAD_ACCEPTED);
            return;
        }
    }

    constexpr bool WINDOW = MODE == REC_VERIFY || MODE == REC_COMMIT_VERIFY;
    extern __shared__ __align__(16) unsigned char rec_dyn_smem[];
    VerSmem<D, IO>& vs = *reinterpret_cast<VerSmem<D, IO>*>(rec_dyn_smem);  // window modes only
    // Staged copies first (the previous window's log rows to commit, then the
    // first block of this window's rows), then the state tile: all in flight together.
    const int nblk = WINDOW ? (L + VWB - 1) / VWB : 0;
    IO bnext{};  // beta logit (raw) of row tid of the next staged block
    if (MODE == REC_COMMIT_VERIFY && acc > 0)
        stage_log_rows<D>(vs.plog, a.prev_log_f, a.W, H, seq, h, 0, min(acc, VWB));
    if (WINDOW) bnext = stage_window_rows<D, IO>(vs.buf[0], a, seq, h, 0, min(L, VWB));

    float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
    const int r0 = warp * RPW, c0 = lane * CPT;
    float s[RPW][CPT];
    load_tile<D>(Sg, r0, c0, s);
    if (MODE == REC_COMMIT_VERIFY && acc > 0) {
        // commit: the same replay expression as kda_commit_kernel, so the
        // committed state has the bits of `acc` serial decodes
        for (int t0 = 0; t0 < acc; t0 += VWB) {
            const int nr = min(VWB, acc - t0);
            if (t0 == 0) {
                ptx::cp_async_wait_prev();  // the log rows (the window rows may still be in flight)
            } else {
                stage_log_rows<D>(vs.plog, a.prev_log_f, a.W, H, seq, h, t0, nr);
                ptx::cp_async_wait_all();
            }
            __syncthreads();
            replay_log_rows<D>(vs.plog, nr, s);
            __syncthreads();  // plog may be refilled
        }
        store_tile<D>(Sg, r0, c0, s);
    }

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
        if (MODE == REC_COMMIT_VERIFY && acc > 0) {
            // committed conv state: the last K-1 rows of [old state; accepted raw rows]
            const IO* praw = static_cast<const IO*>(a.prev_log_raw);
            float old[3], nw[3];
            for (int r = 0; r < K - 1; ++r) old[r] = ldv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch);
            for (int r = 0; r < K - 1; ++r) {
                const int src = acc - (K - 1) + r;  // window row, or < 0: old state row src + K - 1
                nw[r] = src >= 0 ? ldv(praw + ((size_t)seq * a.W + src) * conv_dim + ch) : old[src + K - 1];
            }
            for (int r = 0; r < K - 1; ++r) {
                stv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch, nw[r]);
                sm.win[ring(r - (K - 1))][c] = nw[r];
            }
        } else {
            for (int r = 0; r < K - 1; ++r)
                sm.win[ring(r - (K - 1))][c] = ldv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch);
        }
    }
    for (int i = tid; i < D; i += REC_THREADS) sm.dtb[i] = a.dt_bias[(size_t)h * D + i];
    RowConst rc{a.gate_mode, a.lb, expf(a.A_log[h]), a.l2_eps, a.norm_eps, a.scale, a.norm_w};
    __syncthreads();

    for (int t = 0; t < L; ++t) {
        const size_t row = (size_t)row0 + t;
        const size_t rh = row * H + h;
        const int cur = ring(t);
        float bval, gval;
        if constexpr (WINDOW) {
            // rows of the window from the staged block (t / VWB)
            const int blk = t / VWB, r = t % VWB;
            VerBuf<D, IO>& vb = vs.buf[blk & 1];
            if (r == 0) {
                if (tid < min(VWB, L - blk * VWB)) vb.bv[tid] = Io<IO>::ld(&bnext);
                ptx::cp_async_wait_all();
                __syncthreads();
                // the other buffer's rows are done: prefetch the next block into it
                if (blk + 1 < nblk)
                    bnext = stage_window_rows<D, IO>(vs.buf[(blk + 1) & 1], a, seq, h, (blk + 1) * VWB,
                                                     min(VWB, L - (blk + 1) * VWB));
            }
            for (int c = tid; c < 3 * D; c += REC_THREADS) sm.win[cur][c] = ldv(&vb.rows[r][c / D][c % D]);
            for (int i = tid; i < D; i += REC_THREADS) sm.fr[i] = ldv(&vb.rows[r][3][i]);
            bval = vb.bv[r];
            gval = (g != nullptr && tid < D) ? ldv(&vb.rows[r][4][tid]) : 0.0f;
        } else {
            for (int c = tid; c < 3 * D; c += REC_THREADS) {
                float x;
                if (c < D) x = ldv(q + rh * D + c);
                else if (c < 2 * D) x = ldv(k + rh * D + (c - D));
                else x = ldv(v + rh * D + (c - 2 * D));
                sm.win[cur][c] = x;
            }
            for (int i = tid; i < D; i += REC_THREADS) sm.fr[i] = ldv(f + rh * D + i);
            bval = ldv(b + rh);
            gval = (g != nullptr && tid < D) ? ldv(g + rh * D + tid) : 0.0f;
        }
        __syncthreads();

        const float o = row_step<D>(sm, s, t, K, rc, bval, gval, g != nullptr);
        if (tid < D) store_out(a.out, rh * D + tid, o, a.out_bf16);

        if (MODE == REC_VERIFY || MODE == REC_COMMIT_VERIFY) {
            float* lg = a.log_f + (((size_t)seq * a.W + t) * H + h) * (3 * D);
            if (tid < D) {
                lg[tid] = sm.alpha[tid];
                lg[D + tid] = sm.act[D + tid] * sm.scal[1];
                lg[2 * D + tid] = row_update<D>(sm, tid);
            }
            IO* lr = static_cast<IO*>(a.log_raw) + ((size_t)seq * a.W + t) * conv_dim;
            for (int c = tid; c < 3 * D; c += REC_THREADS) stv(lr + conv_channel<D>(c, h, H), sm.win[cur][c]);
        }
        __syncthreads();
    }

    if (MODE == REC_PREFILL || MODE == REC_DECODE) {
        store_tile<D>(Sg, r0, c0, s);
        // new conv state: the last K-1 raw rows (older ones from the old state)
        for (int c = tid; c < 3 * D; c += REC_THREADS) {
            const int ch = conv_channel<D>(c, h, H);
            for (int r = 0; r < K - 1; ++r)
                stv(cs + ((size_t)slot * (K - 1) + r) * conv_dim + ch, sm.win[ring(L - (K - 1) + r)][c]);
        }
    }
}

// ------------------------------------------------------------------------
// Verify window at dk = dv = 128 with warp-local rows.
//
// The register kernel's thread tiles (16 key dims x 4 value dims, the key
// dims of tile (m, .) being [16m, 16m + 16)) are assigned so that the eight
// tiles of a value-dim block share a warp: warp w holds value dims [16w, +16),
// lane l = 4m + c key dims [16m, +16) of value dims [16w + 4c, +4).  Each
// thread forms the register kernel's partial sums of S'^T k and S^T q over its
// 16 key dims, and their sum over the eight key-dim blocks -- in block order,
// as the register kernel sums its warps -- is read back from a per-warp
// scratch after a warp barrier.  So a row needs no block barrier.  The parts of
// a row that do not depend on the state (conv, SiLU, sums of squares, decay)
// run for a staged block of rows at a time before its rows, and the gated norm
// after them.  Every value is formed by the register kernel's expressions in
// its order, so verified rows, their log and the committed states have the
// bits of decoded rows.

constexpr int VWD = 128;

template <typename IO> struct VwBuf {
    IO rows[VWB][5][VWD];   // q, k, v, f, g of each row of the block
    IO halo[3][3][VWD];     // raw q|k|v rows 3, 2, 1 before the block (before the window: the conv history)
    float bv[VWB];          // beta logits
};

// Key-dim arrays of a row are padded by 4 floats every 16 (index i -> vw_pad(i)),
// so the eight 16-float key-dim blocks a warp reads at once start in distinct
// bank groups (float4 reads without conflicts).
constexpr int VWP = VWD + VWD / 4;
__device__ __forceinline__ int vw_pad(int i) { return i + 4 * (i >> 4); }

template <typename IO> struct VwSmem {
    VwBuf<IO> buf[2];                 // double-buffered staged blocks
    float plog[VWB][3 * VWD];         // log rows to replay (commit first)
    float cw[3 * VWD][4];             // conv taps (K-tap form, oldest first)
    float dtb[VWD];                   // dt_bias of this head
    float qp[VWB][VWP];               // post-SiLU q' of the block's rows (padded key dims)
    float kp[VWB][VWP];               // post-SiLU k' (padded key dims)
    float ap[VWB][VWP];               // decays (padded key dims)
    float vp[VWB][VWD];               // post-SiLU v'
    float nrm[VWB][8];                // per-32-channel sums of squares of q', k'
    float rs[VWB][4];                 // per row: q and k inverse norms, beta
    float o[VWB][VWD];                // outputs before the gated norm
    float esum[VWB][4];               // gated norm: per-32-column sums of squares
    float red[REC_WARPS][8][16];      // per-warp scratch: [key block][value dim] partials of S'^T k
    float red2[REC_WARPS][8][16];     // the same for S^T q
};

// Source of history row r (0 = oldest of the K-1) of the conv state the
// window starts from: the stored conv state, or -- after committing `acc`
// rows of the previous window -- its last K-1 rows of [old state; accepted rows].
template <typename IO>
__device__ __forceinline__ const IO* vw_hist_row(const RecArgs& a, int seq, int slot, int acc, int r, int seg, int h)
{
    const int K = a.K, conv_dim = 3 * a.H * VWD;
    const int src = acc - (K - 1) + r;  // previous window row, or < 0: old state row src + K - 1
    const size_t chan = (size_t)seg * a.H * VWD + (size_t)h * VWD;
    if (src >= 0) return static_cast<const IO*>(a.prev_log_raw) + ((size_t)seq * a.W + src) * conv_dim + chan;
    return static_cast<const IO*>(a.conv_state) + ((size_t)slot * (K - 1) + src + K - 1) * conv_dim + chan;
}

// Issue the copies of window rows [t0, t0 + nr) and of the three raw rows
// before them (all threads; one commit group); window row x is token row
// rbase + x.  Returns the raw beta logit of row t0 + tid (tid < nr), to be
// published in vb.bv with the block.
template <typename IO>
__device__ __forceinline__ IO vw_stage(VwBuf<IO>& vb, const RecArgs& a, int seq, int h, int slot, int acc,
                                       int rbase, int t0, int nr)
{
    constexpr int EPP = 16 / (int)sizeof(IO), PIECES = VWD / EPP;
    const int ntens = a.g != nullptr ? 5 : 4;
    for (int idx = threadIdx.x; idx < nr * ntens * PIECES; idx += REC_THREADS) {
        const int piece = idx % PIECES, rest = idx / PIECES, tens = rest % ntens, r = rest / ntens;
        const size_t rh = ((size_t)rbase + t0 + r) * a.H + h;
        const void* base = tens == 0 ? a.q : tens == 1 ? a.k : tens == 2 ? a.v : tens == 3 ? a.f : a.g;
        ptx::cp_async16(&vb.rows[r][tens][piece * EPP], static_cast<const IO*>(base) + rh * VWD + piece * EPP, 16);
    }
    for (int idx = threadIdx.x; idx < 9 * PIECES; idx += REC_THREADS) {
        const int piece = idx % PIECES, seg = (idx / PIECES) % 3, hr = idx / (3 * PIECES);
        const int x = t0 - 3 + hr;  // window row of this halo row
        const IO* src;
        if (x >= 0) {
            const void* base = seg == 0 ? a.q : seg == 1 ? a.k : a.v;
            src = static_cast<const IO*>(base) + (((size_t)rbase + x) * a.H + h) * VWD;
        } else {
            const int r = x + a.K - 1;  // history row; r < 0: a tap the conv does not have
            if (r < 0) continue;
            src = vw_hist_row<IO>(a, seq, slot, acc, r, seg, h);
        }
        ptx::cp_async16(&vb.halo[hr][seg][piece * EPP], src + piece * EPP, 16);
    }
    ptx::cp_async_commit();
    const IO* b = static_cast<const IO*>(a.b);
    IO braw{};
    if (threadIdx.x < nr) braw = b[((size_t)rbase + t0 + threadIdx.x) * a.H + h];
    return braw;
}

// State-independent part of rows [0, nr) of a staged block for one conv
// channel `it` (q | k | v) of this thread: the register kernel's row_conv
// expressions -- acc = fma(w_j, x_{t-K+1+j}, acc) over j = 0..K-1 from 0,
// SiLU, and for q and k the warp's sum of squares over its 32 consecutive
// channels.  All VWB rows of the block are computed at once (rows past nr
// read whatever the buffer holds and are never stored), so the rows' loads,
// exponentials and shuffle reductions overlap instead of running one row at
// a time; every stored value has the one-row-at-a-time bits.
template <int KK, typename IO>
__device__ __forceinline__ void vw_conv_channel(VwSmem<IO>& sm, const VwBuf<IO>& vb, int it, int nr, int lane)
{
    constexpr int D = VWD;
    const int seg = it / D, ch = it % D;
    float w[KK], xs[KK - 1 + VWB];  // raw rows -(KK-1) .. VWB-1 of the block
#pragma unroll
    for (int j = 0; j < KK; ++j) w[j] = sm.cw[it][j];
#pragma unroll
    for (int j = 0; j + 1 < KK; ++j) xs[j] = ldv(&vb.halo[4 - KK + j][seg][ch]);
#pragma unroll
    for (int t = 0; t < VWB; ++t) xs[KK - 1 + t] = ldv(&vb.rows[t][seg][ch]);
    float x[VWB];
#pragma unroll
    for (int t = 0; t < VWB; ++t) {
        float accv = 0.0f;
#pragma unroll
        for (int j = 0; j < KK; ++j) accv = __fmaf_rn(w[j], xs[t + j], accv);
        x[t] = siluf_(accv);
    }
    if (seg == 2) {
#pragma unroll
        for (int t = 0; t < VWB; ++t)
            if (t < nr) sm.vp[t][ch] = x[t];
    } else {  // warp-uniform: a warp holds 32 consecutive q or k channels
        float(*dst)[VWP] = seg == 0 ? sm.qp : sm.kp;
        float ss[VWB];
#pragma unroll
        for (int t = 0; t < VWB; ++t) ss[t] = warp_sum(x[t] * x[t]);
#pragma unroll
        for (int t = 0; t < VWB; ++t) {
            if (t < nr) {
                dst[t][vw_pad(ch)] = x[t];
                if (lane == 0) sm.nrm[t][it >> 5] = ss[t];
            }
        }
    }
}

template <typename IO>
__device__ __forceinline__ void vw_conv(VwSmem<IO>& sm, const VwBuf<IO>& vb, int K, int it, int nr, int lane)
{
    if (K == 4) vw_conv_channel<4, IO>(sm, vb, it, nr, lane);
    else if (K == 3) vw_conv_channel<3, IO>(sm, vb, it, nr, lane);
    else vw_conv_channel<2, IO>(sm, vb, it, nr, lane);
}

template <typename IO, int MODE>
__global__ void __launch_bounds__(REC_THREADS, 2) kda_verify_warp_kernel(const RecArgs a)
{
    extern __shared__ __align__(16) unsigned char vw_dyn_smem[];
    VwSmem<IO>& sm = *reinterpret_cast<VwSmem<IO>*>(vw_dyn_smem);
    constexpr int D = VWD, RPW = 16, CPT = 4, EPP = 16 / (int)sizeof(IO);
    constexpr bool CV = MODE == REC_COMMIT_VERIFY;
    constexpr bool PF = MODE == REC_PREFILL;  // a whole sequence: no log, the final states stored
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m = lane >> 2, cq = lane & 3;
    const int r0 = RPW * m, c0 = 16 * warp + CPT * cq;  // this thread's tile: key dims [r0, +16), value dims [c0, +4)
    const int H = a.H, K = a.K, W = a.W;
    const int seq = blockIdx.x / H, h = blockIdx.x % H;
    const int conv_dim = 3 * H * D;
    const bool has_g = a.g != nullptr;

    const int slot = a.slots ? a.slots[seq] : seq;
    if (slot < 0) return;  // padding sequence: nothing to do
    if (slot >= a.num_slots) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    int L = W, rbase = seq * W;  // rows of the window (prefill: of the sequence) and the token row of its first
    if (PF) {
        const int s0 = a.cu_seqlens[seq], s1 = a.cu_seqlens[seq + 1];
        if (s0 < 0 || s1 < s0 || s1 > a.T) {
            if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SEQLENS);
            return;
        }
        rbase = s0;
        L = s1 - s0;
        if (L == 0) return;  // zero-length sequence: states unchanged
    }
    int acc = 0;  // commit first: rows of the previous window to replay
    if (CV) {
        acc = a.accepted[seq];
        if (acc < 0 || acc > W) {
            if (tid == 0 && h == 0) flag_status(a.dev_status, KDA_DEV_BAD_ACCEPTED);
            return;
        }
    }

    // staged copies first (the log rows to commit, the first block of rows with
    // the conv history before it), then the parameters and the state tile
    const int nblk = (L + VWB - 1) / VWB;
    if (CV && acc > 0) stage_log_rows<D>(sm.plog, a.prev_log_f, W, H, seq, h, 0, min(acc, VWB));
    IO bnext = vw_stage<IO>(sm.buf[0], a, seq, h, slot, acc, rbase, 0, min(L, VWB));
    for (int c = tid; c < 3 * D; c += REC_THREADS) {
        const int ch = conv_channel<D>(c, h, H);
        for (int j = 0; j < K; ++j) sm.cw[c][j] = a.conv_w[(size_t)ch * K + j];
    }
    for (int i = tid; i < D; i += REC_THREADS) sm.dtb[i] = a.dt_bias[(size_t)h * D + i];
    const RowConst rc{a.gate_mode, a.lb, expf(a.A_log[h]), a.l2_eps, a.norm_eps, a.scale, a.norm_w};

    float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
    float s[RPW][CPT];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const float4 x = ld_stream4(Sg + (size_t)(r0 + rr) * D + c0);
        s[rr][0] = x.x; s[rr][1] = x.y; s[rr][2] = x.z; s[rr][3] = x.w;
    }
    if (CV && acc > 0) {
        // commit: S <- fma(k^, u, alpha * S) per logged row, the decoded row's expression
        for (int t0 = 0; t0 < acc; t0 += VWB) {
            const int nr = min(VWB, acc - t0);
            if (t0 == 0) {
                ptx::cp_async_wait_prev();  // the log rows; the window rows may still be in flight
            } else {
                stage_log_rows<D>(sm.plog, a.prev_log_f, W, H, seq, h, t0, nr);
                ptx::cp_async_wait_all();
            }
            __syncthreads();
            for (int t = 0; t < nr; ++t) {
                const float* lg = sm.plog[t];
                const float4 u4 = *reinterpret_cast<const float4*>(lg + 2 * D + c0);
                const float uc[CPT] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr) {
                    const float ai = lg[r0 + rr], ki = lg[D + r0 + rr];
#pragma unroll
                    for (int cc = 0; cc < CPT; ++cc) s[rr][cc] = __fmaf_rn(ki, uc[cc], __fmul_rn(ai, s[rr][cc]));
                }
            }
            __syncthreads();  // plog may be refilled
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
            st_stream4(Sg + (size_t)(r0 + rr) * D + c0, make_float4(s[rr][0], s[rr][1], s[rr][2], s[rr][3]));
    }

    IO* cs = static_cast<IO*>(a.conv_state);
    IO* lraw = static_cast<IO*>(a.log_raw);
    for (int blk = 0; blk < nblk; ++blk) {
        const int t0 = blk * VWB, nr = min(VWB, L - t0);
        VwBuf<IO>& vb = sm.buf[blk & 1];
        if (tid < nr) vb.bv[tid] = Io<IO>::ld(&bnext);
        ptx::cp_async_wait_all();
        __syncthreads();  // the block is staged; the previous block (rows, epilogue) is done
        if (blk + 1 < nblk)
            bnext = vw_stage<IO>(sm.buf[(blk + 1) & 1], a, seq, h, slot, acc, rbase, t0 + VWB, min(VWB, L - t0 - VWB));

        if (CV && blk == 0 && acc > 0) {
            // the committed conv state: the history rows the window starts from
            for (int idx = tid; idx < 3 * (K - 1) * (D / EPP); idx += REC_THREADS) {
                const int piece = idx % (D / EPP), seg = (idx / (D / EPP)) % 3, r = idx / (3 * (D / EPP));
                *reinterpret_cast<int4*>(cs + ((size_t)slot * (K - 1) + r) * conv_dim + (size_t)seg * H * D + h * D +
                                         piece * EPP) =
                    *reinterpret_cast<const int4*>(&vb.halo[r + 4 - K][seg][piece * EPP]);
            }
        }
        // the raw q|k|v rows of the window into the log
        for (int idx = tid; !PF && idx < nr * 3 * (D / EPP); idx += REC_THREADS) {
            const int piece = idx % (D / EPP), seg = (idx / (D / EPP)) % 3, t = idx / (3 * (D / EPP));
            *reinterpret_cast<int4*>(lraw + ((size_t)rbase + t0 + t) * conv_dim + (size_t)seg * H * D + h * D +
                                     piece * EPP) = *reinterpret_cast<const int4*>(&vb.rows[t][seg][piece * EPP]);
        }
        // ---- state-independent part of the block's rows: conv channels (q, k
        // on every warp, v on warps 0-3) and decays (warps 4-7)
        vw_conv<IO>(sm, vb, K, tid, nr, lane);
        if (tid < D) {
            vw_conv<IO>(sm, vb, K, 2 * D + tid, nr, lane);
        } else {
            const int i = tid - D;
            const float dti = sm.dtb[i];
            float al[VWB];  // all rows of the block at once, as in the conv
#pragma unroll
            for (int t = 0; t < VWB; ++t) al[t] = exp_sfu(log_alpha(rc.gate_mode, rc.lb, rc.ea, ldv(&vb.rows[t][3][i]), dti));
#pragma unroll
            for (int t = 0; t < VWB; ++t)
                if (t < nr) sm.ap[t][vw_pad(i)] = al[t];
        }
        __syncthreads();
        if (tid < nr) {  // the register kernel's norms and beta of row tid
            float sq = 0.0f, sk = 0.0f;
#pragma unroll
            for (int p = 0; p < D / 32; ++p) {
                sq += sm.nrm[tid][p];
                sk += sm.nrm[tid][D / 32 + p];
            }
            sm.rs[tid][0] = rsqrtf(sq + rc.l2_eps);
            sm.rs[tid][1] = rsqrtf(sk + rc.l2_eps);
            sm.rs[tid][2] = sigmoidf_(vb.bv[tid]);
        }
        __syncthreads();
        // decay and normalised key of each row into the log
        for (int e = tid; !PF && e < nr * D; e += REC_THREADS) {
            const int t = e / D, i = e % D;
            float* lg = a.log_f + (((size_t)rbase + t0 + t) * H + h) * (3 * D);
            lg[i] = sm.ap[t][vw_pad(i)];
            lg[D + i] = sm.kp[t][vw_pad(i)] * sm.rs[t][1];
        }

        // ---- the rows: the delta rule on the register state, sums inside the warp
        for (int t = 0; t < nr; ++t) {
            const float4 sc = *reinterpret_cast<const float4*>(&sm.rs[t][0]);
            const float rq = sc.x, rk = sc.y, beta = sc.z;
            float kr[RPW], av[RPW], part[CPT];
#pragma unroll
            for (int u = 0; u < RPW; u += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(&sm.kp[t][vw_pad(r0) + u]);
                const float4 a4 = *reinterpret_cast<const float4*>(&sm.ap[t][vw_pad(r0) + u]);
                const float2 ka = __fmul2_rn(make_float2(k4.x, k4.y), make_float2(rk, rk));
                const float2 kb = __fmul2_rn(make_float2(k4.z, k4.w), make_float2(rk, rk));
                kr[u] = ka.x; kr[u + 1] = ka.y; kr[u + 2] = kb.x; kr[u + 3] = kb.y;
                av[u] = a4.x; av[u + 1] = a4.y; av[u + 2] = a4.z; av[u + 3] = a4.w;
            }
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) part[cc] = 0.0f;
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                const float ai = av[rr];
#pragma unroll
                for (int cc = 0; cc < CPT; cc += 2) {
                    const float2 sp = __fmul2_rn(make_float2(ai, ai), make_float2(s[rr][cc], s[rr][cc + 1]));
                    const float2 pp = __ffma2_rn(sp, make_float2(kr[rr], kr[rr]), make_float2(part[cc], part[cc + 1]));
                    s[rr][cc] = sp.x;
                    s[rr][cc + 1] = sp.y;
                    part[cc] = pp.x;
                    part[cc + 1] = pp.y;
                }
            }
            *reinterpret_cast<float4*>(&sm.red[warp][m][CPT * cq]) = make_float4(part[0], part[1], part[2], part[3]);
            __syncwarp();
            float2 kv01 = make_float2(0.0f, 0.0f), kv23 = kv01;
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {  // key-dim blocks in order
                const float4 r4 = *reinterpret_cast<const float4*>(&sm.red[warp][mb][CPT * cq]);
                kv01 = __fadd2_rn(kv01, make_float2(r4.x, r4.y));
                kv23 = __fadd2_rn(kv23, make_float2(r4.z, r4.w));
            }
            const float4 v4 = *reinterpret_cast<const float4*>(&sm.vp[t][c0]);
            const float2 u01 = __fmul2_rn(make_float2(beta, beta), __fadd2_rn(make_float2(v4.x, v4.y), make_float2(-kv01.x, -kv01.y)));
            const float2 u23 = __fmul2_rn(make_float2(beta, beta), __fadd2_rn(make_float2(v4.z, v4.w), make_float2(-kv23.x, -kv23.y)));
            const float uc[CPT] = {u01.x, u01.y, u23.x, u23.y};
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) part[cc] = 0.0f;
#pragma unroll
            for (int u = 0; u < RPW; u += 4) {  // q^ of the tile's key dims
                const float4 q4 = *reinterpret_cast<const float4*>(&sm.qp[t][vw_pad(r0) + u]);
                const float2 qa = __fmul2_rn(make_float2(q4.x, q4.y), make_float2(rq, rq));
                const float2 qb = __fmul2_rn(make_float2(q4.z, q4.w), make_float2(rq, rq));
                av[u] = qa.x; av[u + 1] = qa.y; av[u + 2] = qb.x; av[u + 3] = qb.y;
            }
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                const float qi = av[rr];
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
            }
            *reinterpret_cast<float4*>(&sm.red2[warp][m][CPT * cq]) = make_float4(part[0], part[1], part[2], part[3]);
            __syncwarp();
            if (m == 0) {
                float2 o01 = make_float2(0.0f, 0.0f), o23 = o01;
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) {
                    const float4 r4 = *reinterpret_cast<const float4*>(&sm.red2[warp][mb][CPT * cq]);
                    o01 = __fadd2_rn(o01, make_float2(r4.x, r4.y));
                    o23 = __fadd2_rn(o23, make_float2(r4.z, r4.w));
                }
                o01 = __fmul2_rn(o01, make_float2(rc.scale, rc.scale));
                o23 = __fmul2_rn(o23, make_float2(rc.scale, rc.scale));
                const size_t rh = ((size_t)rbase + t0 + t) * H + h;
                if (!PF)
                    *reinterpret_cast<float4*>(a.log_f + rh * (3 * D) + 2 * D + c0) =
                        make_float4(uc[0], uc[1], uc[2], uc[3]);
                if (has_g) {
                    *reinterpret_cast<float4*>(&sm.o[t][c0]) = make_float4(o01.x, o01.y, o23.x, o23.y);
                } else {
                    store_out(a.out, rh * D + c0, o01.x, a.out_bf16);
                    store_out(a.out, rh * D + c0 + 1, o01.y, a.out_bf16);
                    store_out(a.out, rh * D + c0 + 2, o23.x, a.out_bf16);
                    store_out(a.out, rh * D + c0 + 3, o23.y, a.out_bf16);
                }
            }
        }

        // ---- sigmoid-gated RMSNorm of the block's outputs (the register kernel's row_out)
        if (has_g) {
            __syncthreads();
            for (int task = warp; task < nr * (D / 32); task += REC_WARPS) {
                const int t = task / (D / 32), p = task % (D / 32);
                const float ov = sm.o[t][32 * p + lane];
                const float ss = warp_sum(ov * ov);
                if (lane == 0) sm.esum[t][p] = ss;
            }
            __syncthreads();
            for (int e = tid; e < nr * D; e += REC_THREADS) {
                const int t = e / D, j = e % D;
                float tot = 0.0f;
#pragma unroll
                for (int p = 0; p < D / 32; ++p) tot += sm.esum[t][p];
                const float r = rsqrtf(tot * (1.0f / D) + rc.norm_eps);
                const float wn = rc.norm_w ? rc.norm_w[j] : 1.0f;
                const float y = sm.o[t][j] * r * wn * sigmoidf_(ldv(&vb.rows[t][4][j]));
                store_out(a.out, (((size_t)rbase + t0 + t) * H + h) * D + j, y, a.out_bf16);
            }
        }
    }

    if (PF) {
        // the final state, and the new conv state: the last K-1 raw rows of
        // [old conv state; sequence], from the last staged block or its halo
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
            st_stream4(Sg + (size_t)(r0 + rr) * D + c0, make_float4(s[rr][0], s[rr][1], s[rr][2], s[rr][3]));
        const int tl = (nblk - 1) * VWB;
        const VwBuf<IO>& vb = sm.buf[(nblk - 1) & 1];
        for (int idx = tid; idx < 3 * (K - 1) * (D / EPP); idx += REC_THREADS) {
            const int piece = idx % (D / EPP), seg = (idx / (D / EPP)) % 3, r = idx / (3 * (D / EPP));
            const int x = L - (K - 1) + r - tl;  // row of the last block; < 0: its halo row x + 3
            const IO* src = x >= 0 ? &vb.rows[x][seg][piece * EPP] : &vb.halo[x + 3][seg][piece * EPP];
            *reinterpret_cast<int4*>(cs + ((size_t)slot * (K - 1) + r) * conv_dim + (size_t)seg * H * D + h * D +
                                     piece * EPP) = *reinterpret_cast<const int4*>(src);
        }
    }
}

// ------------------------------------------------------------------------
// Commit: replay the accepted prefix of a verify window from its log.

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

    // the log rows to replay, staged in blocks of VWB (the first in flight with the state loads)
    __shared__ __align__(16) float plog[VWB][3 * D];
    stage_log_rows<D>(plog, a.log_f, W, H, seq, h, 0, min(acc, VWB));
    float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
    const int r0 = warp * RPW, c0 = lane * CPT;
    float s[RPW][CPT];
    load_tile<D>(Sg, r0, c0, s);
    for (int t0 = 0; t0 < acc; t0 += VWB) {
        const int nr = min(VWB, acc - t0);
        if (t0 > 0) stage_log_rows<D>(plog, a.log_f, W, H, seq, h, t0, nr);
        ptx::cp_async_wait_all();
        __syncthreads();
        replay_log_rows<D>(plog, nr, s);
        __syncthreads();  // plog may be refilled
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

// ------------------------------------------------------------------------
// Streaming commit (D = 128): persistent CTAs, a producer warp and 8 replay
// warps.  The producer bulk-copies each unit's state, its accepted log rows
// and the source rows of its new conv state into a stage; the replay warps
// apply S <- fma(k^, u, alpha * S) row after row -- decode's per-element
// expression -- and leave the state in the stage, from where the producer
// stores it and the conv rows back with bulk copies before the stage takes
// its next unit.  Units with nothing accepted move no data.

constexpr int CMT_WMAX = 16;   // log rows a stage holds (longer windows run kda_commit_kernel)
constexpr int CMT_STAGES = 2;

template <typename IO> struct CmtStage {
    float S[DEC_D * DEC_D];        // the unit's state, row-major (64 KiB)
    float lg[CMT_WMAX][3 * DEC_D]; // accepted log rows: alpha | k^ | u
    IO conv[3][3][DEC_D];          // new conv-state rows [row][q|k|v][channel]
    int slot, acc, head, pad;
};

template <typename IO> struct CmtSmem {
    CmtStage<IO> stage[CMT_STAGES];
    uint64_t full[CMT_STAGES], empty[CMT_STAGES];
};

template <typename IO>
__global__ void __launch_bounds__(DEC_THREADS, 1) kda_commit_stream_kernel(const CommitArgs a)
{
    extern __shared__ __align__(128) unsigned char cmt_smem[];
    CmtSmem<IO>& sm = *reinterpret_cast<CmtSmem<IO>*>(cmt_smem);
    constexpr int D = DEC_D, RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, K = a.K, W = a.W, N = a.B;
    const int conv_dim = 3 * H * D;
    const int units = N * H;
    const int u_begin = (int)(((long long)units * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);

    if (tid == 0) {
        for (int s = 0; s < CMT_STAGES; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.empty[s], REC_WARPS);  // one arrival per replay warp
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // programmatic dependent launch: the prologue may overlap the previous
    // kernel (the verify that wrote the log); data is read only after it completes
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    IO* cs = static_cast<IO*>(a.conv_state);
    const IO* raw = static_cast<const IO*>(a.log_raw);

    if (warp == REC_WARPS) {
        // ---------------- producer
        if (lane != 0) return;
        const uint64_t pol = ptx::policy_evict_first();
        auto write_back = [&](int s, int n) -> bool {
            if (!ptx::mbar_wait(&sm.empty[s], n & 1)) {
                flag_status(a.dev_status, KDA_DEV_TIMEOUT);
                return false;
            }
            const CmtStage<IO>& st = sm.stage[s];
            if (st.acc > 0) {
                ptx::bulk_s2g(a.rec_state + ((size_t)st.slot * H + st.head) * D * D, st.S, D * D * 4);
                for (int r = 0; r < K - 1; ++r)
                    for (int seg = 0; seg < 3; ++seg)
                        ptx::bulk_s2g(cs + ((size_t)st.slot * (K - 1) + r) * conv_dim + (size_t)seg * H * D + st.head * D,
                                      st.conv[r][seg], D * sizeof(IO));
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();  // the stage may be refilled
            }
            return true;
        };
        const int count = u_end - u_begin;
        for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
            const int s = i % CMT_STAGES, n = i / CMT_STAGES;
            if (n > 0 && !write_back(s, n - 1)) return;
            CmtStage<IO>& st = sm.stage[s];
            const int h = u / N, seq = u % N;
            int slot = a.slots ? a.slots[seq] : seq;
            int acc = 0;
            if (slot >= a.num_slots) {
                flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
                slot = -1;
            }
            if (slot >= 0) {
                acc = a.accepted[seq];
                if (acc < 0 || acc > W) {
                    if (h == 0) flag_status(a.dev_status, KDA_DEV_BAD_ACCEPTED);
                    acc = 0;
                }
            }
            // the stage's fields first: the arrival below publishes them with the copies
            st.slot = slot;
            st.acc = acc;
            st.head = h;
            if (acc > 0) {
                const uint32_t rowb = D * sizeof(IO);
                const uint32_t bytes = D * D * 4 + (uint32_t)acc * 3 * D * 4 + (uint32_t)(K - 1) * 3 * rowb;
                asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(ptx::smem_u32(&sm.full[s])),
                             "r"(bytes) : "memory");
                ptx::bulk_g2s_stream(st.S, a.rec_state + ((size_t)slot * H + h) * D * D, D * D * 4, &sm.full[s], pol);
                for (int t = 0; t < acc; ++t)
                    ptx::bulk_g2s(st.lg[t], a.log_f + (((size_t)seq * W + t) * H + h) * (3 * D), 3 * D * 4, &sm.full[s]);
                // the new conv state: the last K-1 rows of [old state; accepted raw rows]
                for (int r = 0; r < K - 1; ++r) {
                    const int src = acc - (K - 1) + r;  // window row, or < 0: old state row src + K - 1
                    for (int seg = 0; seg < 3; ++seg) {
                        const size_t chan = (size_t)seg * H * D + (size_t)h * D;
                        const IO* from = src >= 0 ? raw + ((size_t)seq * W + src) * conv_dim + chan
                                                  : cs + ((size_t)slot * (K - 1) + src + K - 1) * conv_dim + chan;
                        ptx::bulk_g2s(st.conv[r][seg], from, rowb, &sm.full[s]);
                    }
                }
            }
            ptx::mbar_arrive(&sm.full[s]);
        }
        for (int i = count > CMT_STAGES ? count - CMT_STAGES : 0; i < count; ++i)
            if (!write_back(i % CMT_STAGES, i / CMT_STAGES)) return;
        ptx::bulk_wait_all();
        return;
    }

    // ---------------- replay warps (warp w: rows [16w, +16), lane l: columns [4l, +4))
    const int r0 = warp * RPW, c0 = lane * CPT;
    for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
        const int s = i % CMT_STAGES, n = i / CMT_STAGES;
        if (!ptx::mbar_wait(&sm.full[s], n & 1)) {
            if (lane == 0) flag_status(a.dev_status, KDA_DEV_TIMEOUT);
            return;
        }
        CmtStage<IO>& st = sm.stage[s];
        const int acc = st.acc;
        if (acc > 0) {
            float sreg[RPW][CPT];
            load_tile_smem<D>(st.S, r0, c0, sreg);
            for (int t = 0; t < acc; ++t) {
                const float* lg = st.lg[t];
                const float4 u4 = *reinterpret_cast<const float4*>(lg + 2 * D + c0);
                const float uc[CPT] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr) {
                    const float ai = lg[r0 + rr], ki = lg[D + r0 + rr];
#pragma unroll
                    for (int cc = 0; cc < CPT; ++cc) sreg[rr][cc] = __fmaf_rn(ki, uc[cc], __fmul_rn(ai, sreg[rr][cc]));
                }
            }
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr)
                *reinterpret_cast<float4*>(st.S + (r0 + rr) * D + c0) =
                    make_float4(sreg[rr][0], sreg[rr][1], sreg[rr][2], sreg[rr][3]);
            ptx::fence_proxy_async_smem();  // the producer's bulk store reads these writes
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.empty[s]);
    }
}

// ------------------------------------------------------------------------
// launchers




// The window modes stage rows in dynamic shared memory (VerSmem).
template <int D, typename IO, int MODE> static cudaError_t launch_window(const RecArgs& a, int units, cudaStream_t st)
{
    static PerDeviceOnce smem_attr;
    const int smem = (int)sizeof(VerSmem<D, IO>);
    cudaError_t e = smem_attr.run([&](int) {
        return cudaFuncSetAttribute(kda_recurrent_kernel<D, IO, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    kda_recurrent_kernel<D, IO, MODE><<<dim3(units), dim3(REC_THREADS), smem, st>>>(a);
    return cudaGetLastError();
}

// Verify windows at dk = dv = 128: the warp-local kernel (dynamic shared memory VwSmem).
template <typename IO, int MODE> static cudaError_t launch_verify_warp(const RecArgs& a, int units, cudaStream_t st)
{
    static PerDeviceOnce smem_attr;
    const int smem = (int)sizeof(VwSmem<IO>);
    cudaError_t e = smem_attr.run([&](int) {
        return cudaFuncSetAttribute(kda_verify_warp_kernel<IO, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    kda_verify_warp_kernel<IO, MODE><<<dim3(units), dim3(REC_THREADS), smem, st>>>(a);
    return cudaGetLastError();
}

template <int D, typename IO>
static cudaError_t launch_rec_d(int mode, const RecArgs& a, int units, cudaStream_t st)
{
    if constexpr (D == VWD) {
        if (mode == REC_PREFILL) return launch_verify_warp<IO, REC_PREFILL>(a, units, st);
        if (mode == REC_VERIFY) return launch_verify_warp<IO, REC_VERIFY>(a, units, st);
        if (mode == REC_COMMIT_VERIFY) return launch_verify_warp<IO, REC_COMMIT_VERIFY>(a, units, st);
    }
    dim3 grid(units), block(REC_THREADS);
    if (mode == REC_PREFILL) kda_recurrent_kernel<D, IO, REC_PREFILL><<<grid, block, 0, st>>>(a);
    else if (mode == REC_DECODE) kda_recurrent_kernel<D, IO, REC_DECODE><<<grid, block, 0, st>>>(a);
    else if (mode == REC_VERIFY) return launch_window<D, IO, REC_VERIFY>(a, units, st);
    else return launch_window<D, IO, REC_COMMIT_VERIFY>(a, units, st);
    return cudaGetLastError();
}

cudaError_t launch_recurrent(int mode, int io_bf16, const RecArgs& a, int units, cudaStream_t st)
{
    if (units <= 0) return cudaSuccess;
    switch (a.D) {
    case 32: return io_bf16 ? launch_rec_d<32, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<32, float>(mode, a, units, st);
    case 64: return io_bf16 ? launch_rec_d<64, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<64, float>(mode, a, units, st);
    case 128:
        if (mode == REC_DECODE)
            return launch_decode_stream_d128(io_bf16, a, units, st);
        return io_bf16 ? launch_rec_d<128, __nv_bfloat16>(mode, a, units, st) : launch_rec_d<128, float>(mode, a, units, st);
    default: return cudaErrorInvalidValue;
    }
}

static_assert(sizeof(CmtSmem<__nv_bfloat16>) <= 232448, "commit stage buffers exceed shared memory");
static_assert(sizeof(CmtSmem<float>) <= 232448, "commit stage buffers exceed shared memory");

template <typename IO> static cudaError_t launch_commit_stream(const CommitArgs& a, int units, cudaStream_t st)
{
    static PerDeviceOnce smem_attr;
    const int smem = (int)sizeof(CmtSmem<IO>);
    cudaError_t e = smem_attr.run([&](int) {
        return cudaFuncSetAttribute(kda_commit_stream_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    // as many streaming CTAs as the decode kernel (27/32 of the SMs)
    const int cap = sm_count() * 27 / 32 > 0 ? sm_count() * 27 / 32 : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units < cap ? units : cap);
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_commit_stream_kernel<IO>, a);
}

cudaError_t launch_commit(int io_bf16, const CommitArgs& a, cudaStream_t st)
{
    const int units = a.B * a.H;
    if (units <= 0) return cudaSuccess;
    if (a.D == DEC_D && a.W <= CMT_WMAX)
        return io_bf16 ? launch_commit_stream<__nv_bfloat16>(a, units, st) : launch_commit_stream<float>(a, units, st);
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
