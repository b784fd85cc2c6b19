// kda_chunk.cu -- chunked (WY/UT) KDA prefill on tcgen05 tensor cores (sm_103a).
//
// One CTA (256 threads, one per SM) walks one (sequence, head) chain in chunks
// of C = 64 rows, restarting at each segment's first row (TensorFold issue
// #850, Oct 15 comment: prompt rows in chunks from a segment's first row).
// With G_r = sum_{t<=r} log alpha_t inside a chunk (per key dim) and S the
// state at the chunk start, the chunk computes
//     A_rs = beta_r sum_i k_ri k_si e^{G_ri - G_si}   (s < r)
//     P_rs =        sum_i q_ri k_si e^{G_ri - G_si}   (s <= r)
//     T = (I + A)^{-1} ;  W = T Diag(beta)(K o e^G) ;  U' = T Diag(beta) V
//     U = U' - W S ;  O = (Q o e^G) S + P U
//     S <- Diag(e^{G_last}) S + (K o e^{G_last - G})^T U
// which is the gated delta rule unrolled over the chunk (exact in real
// arithmetic).
//
// Tensor cores.  Every product is an M = 128 tcgen05.mma (kind::tf32, fp32
// accumulation in tensor memory) in a transposed form whose M dimension is a
// key or value dim: the state lives in TMEM as S^T (lane = value dim j,
// column = key dim i) and, like U^T, feeds later MMAs straight from TMEM as
// the A operand; B operands are K-major 128-byte-swizzled shared-memory tiles.
//
// Precision.  Outputs are dominated by the most recent rows (o_r ~ P_rr u_r),
// a chain of products whose TF32 operand roundings (2^-11 each) would leave
// the largest outputs ~1e-3 off -- too much for a per-element bound of a few
// thousandths of the output RMS.  So the operands on that chain are split
// into a TF32 high part and a TF32 low part (x = hi + lo to ~2^-22):
//     P (and A)  = [K~; Q~hi] (B1hi + B1lo)^T + [Q~lo; K~] B1hi^T
//     U'         = T (Y + Ylo)                    (Y = Diag(beta) V)
//     P U        = P_hi U_hi + P_hi U_lo + P_lo U_hi
//     K~^T U     = KD_hi U_hi + KD_hi U_lo + KD_lo U_hi   (the state update)
//     (Q o e^G) S = QE_hi S_hi + QE_hi S_lo + QE_lo S_hi  (long prompts: the
//                  carried state dominates the outputs)
// where S_hi is the state as the tensor core reads it from TMEM (fp32 with
// the low 13 mantissa bits dropped) and S_lo = S - S_hi, exact in fp32.  The
// remaining products (W, W S, T) are single TF32 with operands rounded to
// nearest.  The two A operands of the first product share their K~ rows:
// within each 24 KiB K-block the layout is [Q~lo | K~ | Q~hi] (64 rows each),
// and the tiles start at the first and the second 64-row slot.
//
// Range of the decay factors: e^{G} over 64 rows reaches e^{-320}, so A and P
// factor e^{G_r - G_s} around a reference row per 32-row half (row 16 or 48):
// every factor stays in [e^-80, e^80] when each row's log-decay is >= -5 (the
// safe gate with lower bound >= -5); the block of rows r in the second half
// against columns s in the first half uses the second half's reference on
// both sides.  Other gates run on the serial kernel.
//
// TMEM (512 columns): S^T [0,128); X^T [128,192), Y^T [192,256),
// Ylo^T [256,320), D1 [320,416), D1c [416,512) until the first product is
// read; then W^T [320,384), U'^T -> U^T (hi) [384,448), O^T [128,192),
// S^T low part [192,320), U^T low part [448,512).
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace chk {

constexpr int D = 128;
constexpr int C = 64;
constexpr int NT = 256;
constexpr int HALO = 3;
constexpr int RAWR = C + HALO;  // staged raw rows per tensor

constexpr uint32_t TM_ST = 0, TM_XT = 128, TM_YT = 192, TM_YL = 256, TM_D1 = 320, TM_D1C = 416;
constexpr uint32_t TM_WT = 320, TM_UT = 384, TM_OT = 128, TM_SL = 192, TM_UL = 448;
constexpr uint32_t TM_COLS = 512;

// shared memory map (bytes); tiles 1 KiB aligned
constexpr int SM_RAW = 0;                      // q, k, v [67][128] bf16 then f [64][128] bf16
constexpr int RAW_T = RAWR * D * 2;            // 17152 per tensor
constexpr int SM_RAWF = 3 * RAW_T;             // 51456
constexpr int SM_AX = 0;                       // [Q~lo | K~ | Q~hi] x 4 K-blocks of 24 KiB
constexpr int AX_KB = 3 * 64 * 128;            // 24576
constexpr int SM_B1H = 98304;                  // B1 high, 96 rows x 128 K
constexpr int SM_B1L = 147456;                 // B1 low
constexpr int B1_KB = 96 * 128;                // 12288
constexpr int T64_KB = 64 * 128;               // K-block stride of a 64-row tile
constexpr int SM_AKK = 0;                      // A [64][65] fp32 (after the first product)
constexpr int SM_PTMP = 16896;                 // [Q~lo ; K~] B1hi^T part of P [64][65]
constexpr int SM_TS = 33792;                   // solve scratch [64][65]
constexpr int SM_T = 51200;                    // T tile 64 x 64
constexpr int SM_PH = 67584;                   // P high tile 64 x 64
constexpr int SM_PL = 83968;                   // P low tile
constexpr int SM_QE = 100352;                  // Q o e^G tile 64 x 128
constexpr int SM_KD = 133120;                  // (K o e^{G_C - G})^T tile 128 x 64
constexpr int SM_KDL = 165888;                 // low part of the KD tile
constexpr int SM_QEL = 0;                      // low part of the QE tile (after the solve)
constexpr int SM_NW = 33792;                   // -W tile 64 x 128 (after the second product)
constexpr int SM_MISC = 198656;
struct Misc {
    float beta[C];
    float gx[3][D];           // G at rows 31, 48, 63 (per key dim)
    float npart[2][2][4][32]; // q/k row-norm partials [qk][half][warp][row]
    float nrm[2][C];          // q/k inverse norms
    float gamma[D];           // e^{G_C}
    float epart[2][4][32];    // output-norm partials
    float rms[C];
    float M[3][16][16];       // solve scratch
    uint64_t bar;
    uint32_t tmem;
    int err;
};
constexpr int SMEM_BYTES = SM_MISC + (int)sizeof(Misc);
static_assert(SM_RAWF + C * D * 2 <= SM_B1H, "raw staging overlaps B1");
static_assert(SM_AX + 4 * AX_KB <= SM_B1H && SM_B1H + 4 * B1_KB <= SM_B1L && SM_B1L + 4 * B1_KB <= SM_MISC,
              "first-product operands overlap");
static_assert(SM_PTMP >= SM_AKK + 64 * 65 * 4 && SM_TS >= SM_PTMP + 64 * 65 * 4 && SM_T >= SM_TS + 64 * 65 * 4,
              "scratch overlap");
static_assert(SM_PH >= SM_T + 16384 && SM_PL >= SM_PH + 16384 && SM_QE >= SM_PL + 16384 &&
              SM_KD >= SM_QE + 32768 && SM_KDL >= SM_KD + 32768 && SM_KDL + 32768 <= SM_MISC, "tile overlap");
static_assert(SM_QEL + 32768 <= SM_TS && SM_NW >= SM_QEL + 32768 && SM_NW + 32768 <= SM_PH,
              "late tiles overlap");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// byte offset of element (row, k) in a K-major SW128 fp32 tile whose K-blocks
// are `kbs` bytes apart (row 0 of the tile at offset 0)
__device__ __forceinline__ uint32_t swz(int row, int k, int kbs)
{
    return (uint32_t)((k >> 5) * kbs + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + (k & 3) * 4);
}

// Round to the nearest TF32 value (10 explicit mantissa bits).  The tensor
// core would otherwise drop the low mantissa bits of an fp32 operand, a biased
// error twice as large.
__device__ __forceinline__ float tf32r(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void st_raw(unsigned char* sm, uint32_t off, float x)
{
    *reinterpret_cast<float*>(sm + off) = x;
}

// store the TF32 high part of x, or its high and low parts into two tiles
__device__ __forceinline__ void st_hi(unsigned char* sm, uint32_t off, float x) { st_raw(sm, off, tf32r(x)); }
__device__ __forceinline__ void st_hilo(unsigned char* sm, uint32_t off_hi, uint32_t off_lo, float x)
{
    const float hi = tf32r(x);
    st_raw(sm, off_hi, hi);
    st_raw(sm, off_lo, tf32r(x - hi));
}

// Warp transpose-reduction: v[k] (k = 0..31) per lane -> lane l returns the
// sum over the warp's lanes of v[l].  31 shuffles.
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
            const float give = up ? v[k] : v[k + off];
            const float keep = up ? v[k + off] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, give, off);
        }
    }
    return v[0];
}

__device__ __forceinline__ uint64_t dsc(unsigned char* sm, int off)
{
    return ptx::desc_sw128(ptx::smem_u32(sm + off));
}

// One thread waits (bounded) for the next MMA-completion phase and publishes
// the outcome; every thread then passes the barrier and reads the same flag.
__device__ __forceinline__ bool wait_mma(Misc& ms, uint32_t& ph, int32_t* dev_status)
{
    if (threadIdx.x == 0 && !ptx::mbar_wait(&ms.bar, ph)) {
        ms.err = 1;
        flag_status(dev_status, KDA_DEV_TIMEOUT);
    }
    ph ^= 1u;
    __syncthreads();
    ptx::tc_fence_after();
    return ms.err == 0;
}

__global__ void kda_chunk_schedule_kernel(const int32_t* cu, int N, int32_t* order)
{
    for (int s = threadIdx.x; s < N; s += blockDim.x) {
        const int ls = cu[s + 1] - cu[s];
        int rank = 0;
        for (int t = 0; t < N; ++t) {
            const int lt = cu[t + 1] - cu[t];
            rank += (lt > ls) || (lt == ls && t < s);
        }
        order[rank] = s;
    }
}

__global__ void __launch_bounds__(NT, 1) kda_chunk_kernel(const ChunkArgs a)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    Misc& ms = *reinterpret_cast<Misc*>(sm + SM_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = tid & (D - 1);  // channel / key dim / value dim / TMEM lane of this thread
    const int half = tid >> 7;      // chunk rows [32*half, 32*half + 32)
    const int H = a.H, K = a.K;
    const int conv_dim = 3 * H * D;
    const int seq = a.schedule ? a.schedule[blockIdx.x / H] : blockIdx.x / H;
    const int h = blockIdx.x % H;

    // ---- unit checks (before any tensor-memory allocation)
    const int slot = a.slots ? a.slots[seq] : seq;
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    const int seg0 = a.cu_seqlens[seq], seg1 = a.cu_seqlens[seq + 1];
    if (seg0 < 0 || seg1 < seg0 || seg1 > a.T) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_BAD_SEQLENS);
        return;
    }
    if (seg1 == seg0) return;
    if ((ptx::smem_u32(sm) & 1023u) != 0) {  // the 128-byte swizzle assumes 1 KiB-aligned tiles
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_TIMEOUT);
        return;
    }

    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v);
    const __nv_bfloat16* fg = static_cast<const __nv_bfloat16*>(a.f);
    const __nv_bfloat16* bg = static_cast<const __nv_bfloat16*>(a.b);
    const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(a.g);
    __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state);

    if (warp == 0) ptx::tmem_alloc(&ms.tmem, TM_COLS);
    if (tid == 0) {
        ptx::mbar_init(&ms.bar, 1);
        ptx::fence_mbar_init();
        ms.err = 0;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ms.tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter
    const int lrow = (warp & 3) * 32 + lane;                        // TMEM lane of this thread (== col)
    uint32_t ph = 0;

    // ---- per-CTA constants: this thread's conv taps (4-tap form) and gate params
    float wq[4], wk[4], wv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) { wq[j] = 0.f; wk[j] = 0.f; wv[j] = 0.f; }
    for (int j = 0; j < K; ++j) {
        wq[j + 4 - K] = a.conv_w[((size_t)0 * H * D + h * D + col) * K + j];
        wk[j + 4 - K] = a.conv_w[((size_t)1 * H * D + h * D + col) * K + j];
        wv[j + 4 - K] = a.conv_w[((size_t)2 * H * D + h * D + col) * K + j];
    }
    const float dtc = a.dt_bias[(size_t)h * D + col];
    const float ea = expf(a.A_log[h]);
    const float nw = a.norm_w ? a.norm_w[col] : 1.0f;

    // ---- initial state -> TMEM S^T (lane j = col, key dims [64*half, +64))
    {
        const float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = Sg[(size_t)(64 * half + 32 * part + x) * D + col];
            ptx::tmem_st32(tmem + lane_base + TM_ST + 64 * half + 32 * part, v);
        }
    }

    const int nchunks = (seg1 - seg0 + C - 1) / C;
    for (int ch = 0; ch < nchunks && !ms.err; ++ch) {
        const int c0 = seg0 + ch * C;
        const int nvalid = min(C, seg1 - c0);
        const int r0 = 32 * half;

        // ---- stage the raw rows (q, k, v with 3 halo rows; gate f) in shared memory
        for (int idx = tid; idx < 3 * RAWR * 16; idx += NT) {
            const int tsel = idx / (RAWR * 16), rem = idx % (RAWR * 16), sr = rem >> 4, c16 = rem & 15;
            const int gr = c0 - HALO + sr;
            const __nv_bfloat16* base = tsel == 0 ? qg : (tsel == 1 ? kg : vg);
            const void* src = base;
            uint32_t bytes = 0;
            if (gr >= seg0 && gr < seg1) {
                src = base + ((size_t)gr * H + h) * D + c16 * 8;
                bytes = 16;
            } else if (gr < seg0) {
                const int cr = (K - 1) + (gr - seg0);  // conv-state row
                if (cr >= 0) {
                    src = cs + ((size_t)slot * (K - 1) + cr) * conv_dim + (size_t)tsel * H * D + h * D + c16 * 8;
                    bytes = 16;
                }
            }
            ptx::cp_async16(sm + SM_RAW + tsel * RAW_T + sr * (D * 2) + c16 * 16, src, bytes);
        }
        for (int idx = tid; idx < C * 16; idx += NT) {
            const int sr = idx >> 4, c16 = idx & 15, gr = c0 + sr;
            const bool ok = gr < seg1;
            ptx::cp_async16(sm + SM_RAWF + sr * (D * 2) + c16 * 16,
                            ok ? (const void*)(fg + ((size_t)gr * H + h) * D + c16 * 8) : (const void*)fg, ok ? 16 : 0);
        }
        ptx::cp_async_commit();
        if (tid < C) ms.beta[tid] = tid < nvalid ? sigmoidf_(__bfloat162float(bg[(size_t)(c0 + tid) * H + h])) : 0.0f;
        ptx::cp_async_wait_all();
        __syncthreads();

        const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(sm + SM_RAW);
        const __nv_bfloat16* rawf = reinterpret_cast<const __nv_bfloat16*>(sm + SM_RAWF);
        if (ch == nchunks - 1) {
            // the new conv state: the sequence's last K-1 raw rows
            for (int idx = tid; idx < 3 * D * (K - 1); idx += NT) {
                const int r = idx / (3 * D), c = idx % (3 * D), tsel = c / D, cc = c % D;
                const int sr = HALO + nvalid - (K - 1) + r;
                cs[((size_t)slot * (K - 1) + r) * conv_dim + (size_t)tsel * H * D + h * D + cc] =
                    raw[tsel * RAWR * D + sr * D + cc];
            }
        }

        // ---- prep: conv + SiLU, gate, running G for this thread's column and 32 rows
        float qv[32], kv[32], vv[32], G[32];
        {
            float xq[4], xk[4], xv[4];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                xq[j] = __bfloat162float(raw[0 * RAWR * D + (r0 + j) * D + col]);
                xk[j] = __bfloat162float(raw[1 * RAWR * D + (r0 + j) * D + col]);
                xv[j] = __bfloat162float(raw[2 * RAWR * D + (r0 + j) * D + col]);
            }
            float run = 0.0f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int lr = r0 + r;
                xq[3] = __bfloat162float(raw[0 * RAWR * D + (lr + 3) * D + col]);
                xk[3] = __bfloat162float(raw[1 * RAWR * D + (lr + 3) * D + col]);
                xv[3] = __bfloat162float(raw[2 * RAWR * D + (lr + 3) * D + col]);
                float aq = 0.f, ak = 0.f, av = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    aq = __fmaf_rn(wq[j], xq[j], aq);
                    ak = __fmaf_rn(wk[j], xk[j], ak);
                    av = __fmaf_rn(wv[j], xv[j], av);
                }
                const bool ok = lr < nvalid;
                qv[r] = ok ? siluf_(aq) : 0.0f;
                kv[r] = ok ? siluf_(ak) : 0.0f;
                vv[r] = ok ? siluf_(av) : 0.0f;
                const float la = ok ? log_alpha(a.gate_mode, a.lb, ea, __bfloat162float(rawf[lr * D + col]), dtc) : 0.0f;
                run += la;
                G[r] = run;
#pragma unroll
                for (int j = 0; j < 3; ++j) { xq[j] = xq[j + 1]; xk[j] = xk[j + 1]; xv[j] = xv[j + 1]; }
            }
        }
        // row norms of q' and k' (this warp's 32 columns), and the first half's G total
        {
            float t[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) t[r] = qv[r] * qv[r];
            const float pq = transpose_reduce(t, lane);
#pragma unroll
            for (int r = 0; r < 32; ++r) t[r] = kv[r] * kv[r];
            const float pk = transpose_reduce(t, lane);
            ms.npart[0][half][warp & 3][lane] = pq;
            ms.npart[1][half][warp & 3][lane] = pk;
            if (half == 0) ms.gx[0][col] = G[31];
        }
        __syncthreads();
        if (half == 1) {
            const float g31 = ms.gx[0][col];
#pragma unroll
            for (int r = 0; r < 32; ++r) G[r] += g31;
            ms.gx[1][col] = G[16];   // row 48
            ms.gx[2][col] = G[31];   // row 63 (G_C)
            ms.gamma[col] = __expf(G[31]);
        }
        if (tid < 2 * C) {
            const int qk = tid / C, r = tid % C;
            const float tot = ms.npart[qk][r >> 5][0][r & 31] + ms.npart[qk][r >> 5][1][r & 31] +
                              ms.npart[qk][r >> 5][2][r & 31] + ms.npart[qk][r >> 5][3][r & 31];
            ms.nrm[qk][r] = rsqrtf(tot + a.l2_eps);
        }
        __syncthreads();
        // normalise in place: qv, kv now hold q^, k^
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            qv[r] *= ms.nrm[0][r0 + r];
            kv[r] *= ms.nrm[1][r0 + r];
        }

        // ---- operands of the first and second products
        const float Gm = G[16];  // reference row 16 (first half) or 48 (second half)
        {
            const float Gm1 = ms.gx[1][col];
            const float eGm0 = __expf(Gm);  // first half only: e^{G_16} >= e^{-85}
            float xt[32], yt[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int rr = r0 + r;
                const float e = __expf(G[r] - Gm);
                const float ie = __expf(Gm - G[r]);
                const float qq = qv[r] * e;
                // [Q~lo | K~ | Q~hi] slots of 64 rows inside each K-block
                const uint32_t o = swz(rr, col, AX_KB);
                st_hi(sm, SM_AX + 8192 + o, kv[r] * e);
                st_hilo(sm, SM_AX + 16384 + o, SM_AX + o, qq);
                st_hilo(sm, SM_B1H + swz(rr, col, B1_KB), SM_B1L + swz(rr, col, B1_KB), kv[r] * ie);
                if (half == 0)
                    st_hilo(sm, SM_B1H + swz(64 + rr, col, B1_KB), SM_B1L + swz(64 + rr, col, B1_KB),
                            kv[r] * __expf(Gm1 - G[r]));
                const float eG = half == 0 ? e * eGm0 : __expf(G[r]);
                xt[r] = tf32r(ms.beta[rr] * kv[r] * eG);
                yt[r] = ms.beta[rr] * vv[r];
            }
            ptx::tmem_st32(tmem + lane_base + TM_XT + 32 * half, xt);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float hi = tf32r(yt[r]);
                xt[r] = tf32r(yt[r] - hi);
                yt[r] = hi;
            }
            ptx::tmem_st32(tmem + lane_base + TM_YT + 32 * half, yt);
            ptx::tmem_st32(tmem + lane_base + TM_YL + 32 * half, xt);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- first product: D1 = [K~; Q~hi](B1hi + B1lo)^T, D1c = [Q~lo; K~] B1hi^T
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t id = ptx::idesc_tf32(128, 96);
            for (int ks = 0; ks < 16; ++ks) {
                const int ka = (ks >> 2) * AX_KB + (ks & 3) * 32, kb = (ks >> 2) * B1_KB + (ks & 3) * 32;
                ptx::mma_tf32_ss(tmem + TM_D1, dsc(sm, SM_AX + 8192 + ka), dsc(sm, SM_B1H + kb), id, ks > 0);
            }
            for (int ks = 0; ks < 16; ++ks) {
                const int ka = (ks >> 2) * AX_KB + (ks & 3) * 32, kb = (ks >> 2) * B1_KB + (ks & 3) * 32;
                ptx::mma_tf32_ss(tmem + TM_D1, dsc(sm, SM_AX + 8192 + ka), dsc(sm, SM_B1L + kb), id, 1);
            }
            for (int ks = 0; ks < 16; ++ks) {
                const int ka = (ks >> 2) * AX_KB + (ks & 3) * 32, kb = (ks >> 2) * B1_KB + (ks & 3) * 32;
                ptx::mma_tf32_ss(tmem + TM_D1C, dsc(sm, SM_AX + ka), dsc(sm, SM_B1H + kb), id, ks > 0);
            }
            ptx::mma_commit(&ms.bar);
        }
        if (!wait_mma(ms, ph, a.dev_status)) break;

        // ---- A from D1 lanes 0..63; the D1c lanes 0..63 part of P into PTMP.
        // D1 column of (row r, key row s): the first half reads its own block
        // (column s), the second half its own block (column s >= 32) and, for
        // s < 32, the cross block (column 64 + s).  Warps whose lanes are
        // 0..63 (warp & 3 < 2) do this; the branch is warp-uniform.
        if (lrow < 64) {
            float* akk = reinterpret_cast<float*>(sm + SM_AKK);
            float* ptmp = reinterpret_cast<float*>(sm + SM_PTMP);
            const int r = lrow;
            const float br = ms.beta[r];
            float v[32];
            if (half == 0) {
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    ptx::tmem_ld32(tmem + lane_base + TM_D1 + 32 * part, v);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int s = 32 * part + x;
                        if (r < 32 && s >= 32) akk[r * 65 + s] = 0.0f;
                        else if (r < 32 || s >= 32) akk[r * 65 + s] = s < r ? br * v[x] : 0.0f;
                    }
                    ptx::tmem_ld32(tmem + lane_base + TM_D1C + 32 * part, v);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int s = 32 * part + x;
                        if (r < 32 && s >= 32) ptmp[r * 65 + s] = 0.0f;
                        else if (r < 32 || s >= 32) ptmp[r * 65 + s] = v[x];
                    }
                }
            } else {
                ptx::tmem_ld32(tmem + lane_base + TM_D1 + 64, v);
                if (r >= 32) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) akk[r * 65 + x] = br * v[x];
                }
                ptx::tmem_ld32(tmem + lane_base + TM_D1C + 64, v);
                if (r >= 32) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) ptmp[r * 65 + x] = v[x];
                }
            }
        }
        __syncthreads();
        // ---- P = D1 lanes 64..127 + PTMP, masked to s <= r, as high and low tiles
        if (lrow >= 64) {
            const float* ptmp = reinterpret_cast<const float*>(sm + SM_PTMP);
            const int r = lrow - 64;
            float v[32];
            if (half == 0) {
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    ptx::tmem_ld32(tmem + lane_base + TM_D1 + 32 * part, v);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int s = 32 * part + x;
                        if (r < 32 && s >= 32) {
                            st_raw(sm, SM_PH + swz(r, s, T64_KB), 0.0f);
                            st_raw(sm, SM_PL + swz(r, s, T64_KB), 0.0f);
                        } else if (r < 32 || s >= 32) {
                            const float p = s <= r ? v[x] + ptmp[r * 65 + s] : 0.0f;
                            st_hilo(sm, SM_PH + swz(r, s, T64_KB), SM_PL + swz(r, s, T64_KB), p);
                        }
                    }
                }
            } else {
                ptx::tmem_ld32(tmem + lane_base + TM_D1 + 64, v);
                if (r >= 32) {
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        st_hilo(sm, SM_PH + swz(r, x, T64_KB), SM_PL + swz(r, x, T64_KB), v[x] + ptmp[r * 65 + x]);
                }
            }
        }
        // ---- Q o e^G and (K o e^{G_C - G})^T tiles for the later products
        float qe[32];  // q^ e^G, whose low part is stored after the solve
        {
            const float GC = ms.gx[2][col];
            const float eGm0 = __expf(Gm);
            const float cGCm1 = __expf(GC - Gm);  // second half: e^{G_63 - G_48} >= e^{-75}
            float kd[32], kl[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int rr = r0 + r;
                float eG, edec;
                if (half == 0) {
                    eG = __expf(G[r] - Gm) * eGm0;
                    edec = __expf(GC - G[r]);
                } else {
                    eG = __expf(G[r]);
                    edec = __expf(Gm - G[r]) * cGCm1;
                }
                qe[r] = qv[r] * eG;
                st_hi(sm, SM_QE + swz(rr, col, T64_KB), qe[r]);
                const float x = kv[r] * edec;
                kd[r] = tf32r(x);
                kl[r] = tf32r(x - kd[r]);
            }
#pragma unroll
            for (int qd = 0; qd < 8; ++qd) {
                const uint32_t o = half * 128 * 128 + col * 128 + ((qd ^ (col & 7)) << 4);
                *reinterpret_cast<float4*>(sm + SM_KD + o) =
                    make_float4(kd[4 * qd], kd[4 * qd + 1], kd[4 * qd + 2], kd[4 * qd + 3]);
                *reinterpret_cast<float4*>(sm + SM_KDL + o) =
                    make_float4(kl[4 * qd], kl[4 * qd + 1], kl[4 * qd + 2], kl[4 * qd + 3]);
            }
        }
        ptx::tc_fence_before();
        __syncthreads();

        // ---- T = (I + A)^{-1}: 16x16 diagonal blocks, then off-diagonal blocks by level
        {
            const float* akk = reinterpret_cast<const float*>(sm + SM_AKK);
            float* ts = reinterpret_cast<float*>(sm + SM_TS);
            for (int idx = tid; idx < C * 65; idx += NT) ts[idx] = 0.0f;
            __syncthreads();
            if (tid < C) {
                const int bb = tid >> 4, cc = tid & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float accv = (i == cc) ? 1.0f : 0.0f;
#pragma unroll
                    for (int j = 0; j < i; ++j) accv = __fmaf_rn(-akk[(16 * bb + i) * 65 + 16 * bb + j], x[j], accv);
                    x[i] = accv;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) ts[(16 * bb + i) * 65 + 16 * bb + cc] = x[i];
            }
            __syncthreads();
            for (int d = 1; d <= 3; ++d) {
                const int nb = 4 - d;
                for (int idx = tid; idx < nb * 256; idx += NT) {
                    const int bj = idx >> 8, x = (idx >> 4) & 15, y = idx & 15, bi = bj + d;
                    float accv = 0.0f;
                    for (int kk = bj; kk < bi; ++kk)
#pragma unroll
                        for (int z = 0; z < 16; ++z)
                            accv = __fmaf_rn(akk[(16 * bi + x) * 65 + 16 * kk + z], ts[(16 * kk + z) * 65 + 16 * bj + y], accv);
                    ms.M[bj][x][y] = accv;
                }
                __syncthreads();
                for (int idx = tid; idx < nb * 256; idx += NT) {
                    const int bj = idx >> 8, x = (idx >> 4) & 15, y = idx & 15, bi = bj + d;
                    float accv = 0.0f;
#pragma unroll
                    for (int z = 0; z < 16; ++z) accv = __fmaf_rn(ts[(16 * bi + x) * 65 + 16 * bi + z], ms.M[bj][z][y], accv);
                    ts[(16 * bi + x) * 65 + 16 * bj + y] = -accv;
                }
                __syncthreads();
            }
            for (int idx = tid; idx < C * C; idx += NT) {
                const int r = idx / C, s = idx % C;
                st_hi(sm, SM_T + swz(r, s, T64_KB), ts[r * 65 + s]);
            }
        }
        // the low part of the QE tile (over the dead A and P scratch)
#pragma unroll
        for (int r = 0; r < 32; ++r) st_hi(sm, SM_QEL + swz(r0 + r, col, T64_KB), qe[r] - tf32r(qe[r]));
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- second product: W^T = X^T T^T, U'^T = (Y + Ylo)^T T^T
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t id = ptx::idesc_tf32(128, 64);
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t bd = dsc(sm, SM_T + (ks >> 2) * T64_KB + (ks & 3) * 32);
                ptx::mma_tf32_ts(tmem + TM_WT, tmem + TM_XT + ks * 8, bd, id, ks > 0);
                ptx::mma_tf32_ts(tmem + TM_UT, tmem + TM_YT + ks * 8, bd, id, ks > 0);
                ptx::mma_tf32_ts(tmem + TM_UT, tmem + TM_YL + ks * 8, bd, id, 1);
            }
            ptx::mma_commit(&ms.bar);
        }
        if (!wait_mma(ms, ph, a.dev_status)) break;

        // ---- -W tile from W^T (lane i = col, rows 32*half .. +32); S_lo = S - S_hi
        {
            float v[32];
            ptx::tmem_ld32(tmem + lane_base + TM_WT + 32 * half, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) st_hi(sm, SM_NW + swz(32 * half + x, col, T64_KB), -v[x]);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                ptx::tmem_ld32(tmem + lane_base + TM_ST + 64 * half + 32 * part, v);
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] -= __uint_as_float(__float_as_uint(v[x]) & 0xFFFFE000u);
                ptx::tmem_st32(tmem + lane_base + TM_SL + 64 * half + 32 * part, v);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- third product: U^T = U'^T - S^T W^T ; O^T = S^T (Q o e^G)^T (split)
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t id = ptx::idesc_tf32(128, 64);
            for (int ks = 0; ks < 16; ++ks) {
                const int kb = (ks >> 2) * T64_KB + (ks & 3) * 32;
                ptx::mma_tf32_ts(tmem + TM_UT, tmem + TM_ST + ks * 8, dsc(sm, SM_NW + kb), id, 1);
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_ST + ks * 8, dsc(sm, SM_QE + kb), id, ks > 0);
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_SL + ks * 8, dsc(sm, SM_QE + kb), id, 1);
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_ST + ks * 8, dsc(sm, SM_QEL + kb), id, 1);
            }
            ptx::mma_commit(&ms.bar);
        }
        if (!wait_mma(ms, ph, a.dev_status)) break;

        // ---- S^T <- S^T Diag(e^{G_C}); U^T -> high part in place and low part
        {
            float v[32];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t ta = tmem + lane_base + TM_ST + 64 * half + 32 * part;
                ptx::tmem_ld32(ta, v);
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] *= ms.gamma[64 * half + 32 * part + x];
                ptx::tmem_st32(ta, v);
            }
            float lo[32];
            ptx::tmem_ld32(tmem + lane_base + TM_UT + 32 * half, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const float hi = tf32r(v[x]);
                lo[x] = tf32r(v[x] - hi);
                v[x] = hi;
            }
            ptx::tmem_st32(tmem + lane_base + TM_UT + 32 * half, v);
            ptx::tmem_st32(tmem + lane_base + TM_UL + 32 * half, lo);
        }
        ptx::tc_fence_before();
        __syncthreads();

        // ---- fourth product: O^T += U^T P^T ; S^T += U^T (K o e^{G_C - G}) (both split)
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint32_t id64 = ptx::idesc_tf32(128, 64), id128 = ptx::idesc_tf32(128, 128);
            for (int ks = 0; ks < 8; ++ks) {
                const int kb = (ks >> 2) * T64_KB + (ks & 3) * 32;
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_UT + ks * 8, dsc(sm, SM_PH + kb), id64, 1);
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_UL + ks * 8, dsc(sm, SM_PH + kb), id64, 1);
                ptx::mma_tf32_ts(tmem + TM_OT, tmem + TM_UT + ks * 8, dsc(sm, SM_PL + kb), id64, 1);
            }
            for (int ks = 0; ks < 8; ++ks) {
                const int kb = (ks >> 2) * 128 * 128 + (ks & 3) * 32;
                ptx::mma_tf32_ts(tmem + TM_ST, tmem + TM_UT + ks * 8, dsc(sm, SM_KD + kb), id128, 1);
                ptx::mma_tf32_ts(tmem + TM_ST, tmem + TM_UL + ks * 8, dsc(sm, SM_KD + kb), id128, 1);
                ptx::mma_tf32_ts(tmem + TM_ST, tmem + TM_UT + ks * 8, dsc(sm, SM_KDL + kb), id128, 1);
            }
            ptx::mma_commit(&ms.bar);
        }
        if (!wait_mma(ms, ph, a.dev_status)) break;

        // ---- outputs (lane j = col, rows 32*half .. +32), optional gated RMSNorm
        {
            float o[32];
            ptx::tmem_ld32(tmem + lane_base + TM_OT + 32 * half, o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= a.scale;
            if (gg != nullptr) {
                float t[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) t[x] = o[x] * o[x];
                ms.epart[half][warp & 3][lane] = transpose_reduce(t, lane);
                __syncthreads();
                if (tid < C) {
                    const int r = tid;
                    const float tot = ms.epart[r >> 5][0][r & 31] + ms.epart[r >> 5][1][r & 31] +
                                      ms.epart[r >> 5][2][r & 31] + ms.epart[r >> 5][3][r & 31];
                    ms.rms[r] = rsqrtf(tot * (1.0f / D) + a.norm_eps);
                }
                __syncthreads();
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const int r = r0 + x;
                    if (r < nvalid) {
                        const float gv = __bfloat162float(gg[((size_t)(c0 + r) * H + h) * D + col]);
                        o[x] = o[x] * ms.rms[r] * nw * sigmoidf_(gv);
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const int r = r0 + x;
                if (r < nvalid) store_out(a.out, ((size_t)(c0 + r) * H + h) * D + col, o[x], a.out_bf16);
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
    }

    // ---- final state S^T -> rec_state (S[i][j], lane j = col)
    if (!ms.err) {
        float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            ptx::tmem_ld32(tmem + lane_base + TM_ST + 64 * half + 32 * part, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) Sg[(size_t)(64 * half + 32 * part + x) * D + col] = v[x];
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace chk

bool chunk_supported(const kda_params* p)
{
    // dk = dv = 128, bf16 rows, and per-row log decay >= -5 (safe gate, lb >= -5),
    // which keeps every factored decay inside fp32 range
    return p->head_dim_k == 128 && p->head_dim_v == 128 && p->io_dtype == KDA_DTYPE_BF16 &&
           p->gate_mode == KDA_GATE_SAFE && p->gate_lower_bound >= -5.0f;
}

cudaError_t launch_chunk(int io_bf16, const ChunkArgs& a, cudaStream_t st)
{
    if (!io_bf16) return cudaErrorNotSupported;
    static bool attr_done[128];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(chk::kda_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             chk::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    if (a.schedule) chk::kda_chunk_schedule_kernel<<<1, 256, 0, st>>>(a.cu_seqlens, a.N, a.schedule);
    chk::kda_chunk_kernel<<<a.N * a.H, chk::NT, chk::SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
