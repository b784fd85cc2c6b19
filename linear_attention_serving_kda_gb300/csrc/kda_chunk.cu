// kda_chunk.cu -- chunked (WY/UT) KDA prefill on tcgen05 tensor cores (sm_103a).
//
// One CTA (512 threads, one per SM) walks one (sequence, head) chain in chunks
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
// Tensor cores.  Every product is an M = 128 tcgen05.mma (fp32 accumulation
// in tensor memory) in a transposed form whose M dimension is a key or value
// dim: the state lives in TMEM as S^T (lane = value dim j, column = key dim i)
// and, like U^T, feeds later MMAs straight from TMEM as the A operand; B
// operands are K-major 128-byte-swizzled shared-memory tiles.
//
// Precision.  Outputs are dominated by the most recent rows (o_r ~ P_rr u_r),
// a chain of products whose TF32 operand roundings (2^-11 each) would leave
// the largest outputs ~1e-3 off -- too much for a per-element bound of a few
// thousandths of the output RMS.  So the operands on that chain are split.
// The first two products run on tf32 (kind::tf32): the high part is x itself
// as the tensor core reads it (the low 13 mantissa bits dropped) and the low
// part the exact remainder, itself read truncated (x = hi + lo to within
// 2^-20 |x|):
//     P (and A)  = [K~; Q~hi] (B1hi + B1lo)^T + [Q~lo; K~] B1hi^T
//     U'         = T (Y + Ylo)                    (Y = Diag(beta) V)
// with W = X T single TF32 (operands rounded to nearest).  The third and
// fourth products run on bf16 (kind::f16: 16 K elements per MMA, half the
// MMA chain of each accumulator): every operand is split into bf16 high and
// low parts (x = hi + lo to within 2^-16 |x|) and a product sums hi*hi +
// hi*lo + lo*hi:
//     U = U' - W S,  (Q o e^G) S   (S^T split in TMEM; -W, Q o e^G tiles)
//     P U,  (K o e^{G_C - G})^T U  (U^T split in TMEM; P, KD tiles)
// The two A operands of the first product share their K~ rows: within each
// 24 KiB K-block the layout is [Q~lo | K~ | Q~hi] (64 rows each),
// and the tiles start at the first and the second 64-row slot.
//
// Range of the decay factors: e^{G} over 64 rows reaches e^{-320}, so A and P
// factor e^{G_r - G_s} around a reference row per 32-row half (row 16 or 48):
// every factor stays in [e^-80, e^80] when each row's log-decay is >= -5 (the
// safe gate with lower bound >= -5); the block of rows r in the second half
// against columns s in the first half uses the second half's reference on
// both sides.  With other gates (softplus, lower bound < -5) a chunk ends
// before the first row that would take a factor out of that range (chunk_cut),
// so chunk boundaries follow the decays; the next chunk starts there.
//
// TMEM (512 columns): S^T [0,128); X^T [128,192), Y^T [192,256),
// Ylo^T [256,320), D1 [320,416), D1c [416,512) until the first product is
// read; then W^T [320,384), U'^T -> U^T [384,448), O^T [128,192), S^T high
// and low bf16 pairs [192,256), [256,320), U^T high and low pairs [448,480),
// [480,512).
//
// Staging.  A chunk's raw rows (q, k, v with the three rows before it, and
// the gate rows) arrive as four 2-D tensor copies issued by one thread, the
// next chunk's while the current one finishes; a segment's first chunk takes
// its three earlier rows from the conv state instead.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace chk {

constexpr int D = 128;
constexpr int C = 64;
constexpr int NT = 512;         // 16 warps: thread (column c, quarter q) owns rows [16q, 16q+16) of column c
constexpr int RPT = 16;         // rows per thread
constexpr int HALO = 3;
constexpr int RAWR = C + HALO;  // staged raw rows per tensor

constexpr uint32_t TM_ST = 0, TM_XT = 128, TM_YT = 192, TM_YL = 256, TM_D1 = 320, TM_D1C = 416;
constexpr uint32_t TM_WT = 320, TM_UT = 384, TM_OT = 128;
constexpr uint32_t TM_COLS = 512;

// shared memory map (bytes); tiles 1 KiB aligned
constexpr int SM_RAW = 0;                      // q, k, v [67][128] bf16 then f [64][128] bf16
constexpr int RAW_T = RAWR * D * 2;            // 17152 per tensor
constexpr int SM_RAWF = 3 * RAW_T;             // 51456
constexpr int RAW_END = SM_RAWF + C * D * 2;   // 67840
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
constexpr int SM_PH = 68608;                   // P high tile 64 x 64
constexpr int SM_PL = 84992;                   // P low tile
constexpr int SM_QE = 101376;                  // Q o e^G tile 64 x 128
constexpr int SM_KD = 134144;                  // (K o e^{G_C - G})^T tile 128 x 64
constexpr int SM_KDL = 166912;                 // low part of the KD tile
constexpr int SM_MISC = 199680;
struct Misc {
    float beta[C];
    float gq[4][D];           // per-quarter totals of log alpha (per key dim)
    float gx[3][D];           // G at rows 16, 48, 63
    float npart[2][4][4][16]; // q/k row-norm partials [qk][quarter][lane quarter][row]
    float nrm[2][C];          // q/k inverse norms
    float gamma[D];           // e^{G_C}
    float epart[4][4][16];    // output-norm partials [quarter][lane quarter][row]
    float rms[C];
    float X[32][33];          // solve scratch: A[H1,H0] inv(H0)
    uint64_t bar;             // tensor-core completion
    uint64_t rbar;            // raw-row copies (split chain: third-product operands)
    uint64_t bbar;            // split chain: fourth-product operands
    uint32_t tmem;
    int err;
    int ncut;                 // unbounded gates: first row that leaves the factored range
    int staged_t;             // split producers: the task whose rows are staged ahead (-1: none)
    int rows_pending;         // split producers: a row staging in flight, not yet waited for
    int next_ok;              // split producers: the staged task's slot is known to be free
    float beta_next[C];       // split producers: the staged task's beta
    float ganc[2][D];         // unbounded gates: G at rows 0 and 32; then G at the chunk's last row
};
constexpr int SMEM_BYTES = SM_MISC + (int)sizeof(Misc);
static_assert(RAW_END <= SM_B1H && RAW_END <= SM_PH, "raw staging overlaps B1 or the P tiles");
static_assert(SM_AX + 4 * AX_KB <= SM_B1H && SM_B1H + 4 * B1_KB <= SM_B1L && SM_B1L + 4 * B1_KB <= SM_MISC,
              "first-product operands overlap");
static_assert(SM_PTMP >= SM_AKK + 64 * 65 * 4 && SM_TS >= SM_PTMP + 64 * 65 * 4 && SM_T >= SM_TS + 64 * 65 * 4,
              "scratch overlap");
static_assert(SM_PH >= SM_T + 16384 && SM_PL >= SM_PH + 16384 && SM_QE >= SM_PL + 16384 &&
              SM_KD >= SM_QE + 32768 && SM_KDL >= SM_KD + 32768 && SM_KDL + 32768 <= SM_MISC, "tile overlap");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(offsetof(Misc, gamma) % 16 == 0 && SM_MISC % 16 == 0, "e^{G_C} is read as float4");
static_assert(offsetof(Misc, rms) % 8 == 0, "row inverse norms are read as float2");

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

// store the TF32 value nearest to x (an operand used unsplit)
__device__ __forceinline__ void st_hi(unsigned char* sm, uint32_t off, float x) { st_raw(sm, off, tf32r(x)); }



// Warp transpose-reduction of 16 values per lane: lane l returns the sum over
// all 32 lanes of v[l & 15].  16 shuffles.
__device__ __forceinline__ float transpose_reduce16(float (&v)[16], int lane)
{
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
            const float give = up ? v[k] : v[k + off];
            const float keep = up ? v[k + off] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, give, off);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
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

// rows of unit sequence s (a transfer run, s >= nsplit > 0, covers sequence s - nsplit)
__device__ __forceinline__ int unit_rows_seq(int s, int nsplit) { return (nsplit > 0 && s >= nsplit) ? s - nsplit : s; }

__global__ void kda_chunk_schedule_kernel(const int32_t* cu, int N, int nsplit, int32_t* order)
{
    for (int s = threadIdx.x; s < N; s += blockDim.x) {
        const int rs = unit_rows_seq(s, nsplit);
        const int ls = cu[rs + 1] - cu[rs];
        int rank = 0;
        for (int t = 0; t < N; ++t) {
            const int rt = unit_rows_seq(t, nsplit);
            const int lt = cu[rt + 1] - cu[rt];
            rank += (lt > ls) || (lt == ls && t < s);
        }
        order[rank] = s;
    }
}

// Issue the cp.async copies of one chunk's raw rows (q, k, v with 3 halo rows,
// the first chunk's halo from the conv state; gate rows); zero beyond the segment.
// Tensor maps of the raw rows: q, k, v and the gate f, each viewed as a
// [T][H * 128] bf16 matrix; boxes of 128 channels x (C + HALO) rows (C for f).
struct RawMaps {
    CUtensorMap q, k, v, f;
};

// Issue the copies of the raw rows of the chunk starting at row c0 of head h
// (one thread).  Rows past the end of the tensor read as zero; rows past the
// segment's end are read but never used.
__device__ __forceinline__ void stage_chunk(unsigned char* sm, const RawMaps& m, Misc& ms, int c0, int h)
{
    const uint64_t pol = ptx::policy_evict_first();  // rows are read once (and the halo twice)
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive_expect_tx(&ms.rbar, 3 * RAW_T + C * D * 2);
    ptx::tma_load_2d(sm + SM_RAW, &m.q, h * D, c0 - HALO, &ms.rbar, pol);
    ptx::tma_load_2d(sm + SM_RAW + RAW_T, &m.k, h * D, c0 - HALO, &ms.rbar, pol);
    ptx::tma_load_2d(sm + SM_RAW + 2 * RAW_T, &m.v, h * D, c0 - HALO, &ms.rbar, pol);
    ptx::tma_load_2d(sm + SM_RAWF, &m.f, h * D, c0, &ms.rbar, pol);
}

// ---- bf16 operands of the third and fourth products.  Each operand x is
// split into bf16 high and low parts (x = hi + lo to within 2^-16 |x|) and a
// product sums hi*hi + hi*lo + lo*hi in fp32 (kind::f16): 16 K elements per
// MMA halve each accumulator's chain of MMAs against tf32.  Tiles are K-major
// and 128-byte swizzled with 64 bf16 per row; in tensor memory an A operand
// holds two bf16 per 32-bit column, the even k in the low half.
constexpr uint32_t BT64_KB = 8192;   // K-block stride of a 64-row bf16 tile
constexpr uint32_t BT128_KB = 16384; // K-block stride of a 128-row bf16 tile

// shared-memory offsets of the high and low tiles: -W and Q o e^G (64 rows x
// 128 key dims), P (64 x 64), (K o e^{G_C - G})^T (128 key dims x 64 rows)
struct Bf16Tiles {
    uint32_t nwh, nwl, qeh, qel, ph, pl, kdh, kdl;
};
// tensor-memory columns: S^T (fp32), S^T high and low (bf16 pairs), U^T (fp32),
// U^T high and low (bf16 pairs)
struct Bf16Tmem {
    uint32_t st, sh, sl, ut, uh, ul;
};
// the fused kernel's tiles (-W in the region of the first product's low B tile,
// dead after it; the others in the regions of the fp32 tiles they replace, so
// the raw-row staging region is free once the second product has read T) and
// columns (S^T pairs over the dead Y^T / Ylo^T, U^T pairs after U^T)
constexpr uint32_t TM_SH = 192, TM_SL16 = 256, TM_UH = 448, TM_UL16 = 480;
constexpr Bf16Tiles FUSED_TILES{SM_KDL, SM_KDL + 16384, SM_QE, SM_QE + 16384, SM_PH, SM_PH + 8192, SM_KD, SM_KD + 16384};
// the split path's producers publish these tiles while the next task's rows
// are staged below them
static_assert(RAW_END <= FUSED_TILES.ph && RAW_END <= FUSED_TILES.qeh && RAW_END <= FUSED_TILES.kdh &&
                  RAW_END <= FUSED_TILES.nwh,
              "published tiles overlap the raw-row staging region");
constexpr Bf16Tmem FUSED_TMEM{TM_ST, TM_SH, TM_SL16, TM_UT, TM_UH, TM_UL16};
static_assert(SM_KDL % 1024 == 0 && SM_QE % 1024 == 0 && SM_PH % 1024 == 0 && SM_KD % 1024 == 0,
              "bf16 tiles need 1 KiB-aligned bases");
static_assert(SM_KDL + 32768 <= SM_MISC && SM_KD + 32768 <= SM_KDL && RAW_END <= SM_PH,
              "-W (the low K-block region) and the staging region are free after the second product");

// byte offset of bf16 element (row, k) in a K-major SW128 bf16 tile (64 per
// 128-byte row) whose K-blocks are `kbs` bytes apart
__device__ __forceinline__ uint32_t swz16(int row, int k, int kbs)
{
    return (uint32_t)((k >> 6) * kbs + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
}

// bf16 high and low parts of (x0, x1) as packed pairs (x0 in the low half):
// hi = RN(x), lo = RN(x - hi); x - hi is exact in fp32
__device__ __forceinline__ void bf16_split2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// S^T -> bf16 high and low pairs (this thread's 32 key dims)
__device__ __forceinline__ void state_split16(uint32_t t_st, uint32_t t_sh, uint32_t t_sl)
{
    float s[32];
    ptx::tmem_ld32(t_st, s);
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) bf16_split2(s[2 * x], s[2 * x + 1], hi[x], lo[x]);
    ptx::tmem_st16u(t_sh, hi);
    ptx::tmem_st16u(t_sl, lo);
}

// S^T <- S^T Diag(gamma); U^T -> bf16 high and low pairs (this thread's 16 rows)
__device__ __forceinline__ void rescale_split16(uint32_t t_st, uint32_t t_ut, uint32_t t_uh, uint32_t t_ul,
                                                const float* gam32)
{
    float v[32];
    ptx::tmem_ld32(t_st, v);
#pragma unroll
    for (int x = 0; x < 32; x += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gam32 + x);
        const float2 a2 = __fmul2_rn(make_float2(v[x], v[x + 1]), make_float2(g4.x, g4.y));
        const float2 b2 = __fmul2_rn(make_float2(v[x + 2], v[x + 3]), make_float2(g4.z, g4.w));
        v[x] = a2.x; v[x + 1] = a2.y; v[x + 2] = b2.x; v[x + 3] = b2.y;
    }
    ptx::tmem_st32(t_st, v);
    float u[RPT];
    ptx::tmem_ld16(t_ut, u);
    uint32_t hi[RPT / 2], lo[RPT / 2];
#pragma unroll
    for (int x = 0; x < RPT / 2; ++x) bf16_split2(u[2 * x], u[2 * x + 1], hi[x], lo[x]);
    ptx::tmem_st8(t_uh, hi);
    ptx::tmem_st8(t_ul, lo);
}

// -W as bf16 high and low tiles from W^T: this thread's 16 rows of key dim col
__device__ __forceinline__ void store_neg_w16(unsigned char* sm, const Bf16Tiles tl, uint32_t t_wt, int qq, int col)
{
    float w[RPT];
    ptx::tmem_ld16(t_wt, w);
#pragma unroll
    for (int x = 0; x < RPT; x += 2) {
        uint32_t hi, lo;
        bf16_split2(-w[x], -w[x + 1], hi, lo);
        const uint32_t o0 = swz16(RPT * qq + x, col, BT64_KB), o1 = swz16(RPT * qq + x + 1, col, BT64_KB);
        *reinterpret_cast<uint16_t*>(sm + tl.nwh + o0) = (uint16_t)(hi & 0xFFFFu);
        *reinterpret_cast<uint16_t*>(sm + tl.nwh + o1) = (uint16_t)(hi >> 16);
        *reinterpret_cast<uint16_t*>(sm + tl.nwl + o0) = (uint16_t)(lo & 0xFFFFu);
        *reinterpret_cast<uint16_t*>(sm + tl.nwl + o1) = (uint16_t)(lo >> 16);
    }
}

// third product: U^T += S^T (-W)^T (issuer 0) and O^T = S^T (Q o e^G)^T
// (issuer 1), all 64 chunk rows each (few large MMAs: each accumulator's MMAs
// are a chain in one thread); three bf16 terms per K step.
template <int UNR>
__device__ __forceinline__ void issue_third16(unsigned char* sm, uint32_t tmem, int q, const Bf16Tiles tl,
                                              const Bf16Tmem tm, uint32_t c_ot, uint64_t* bar)
{
    ptx::tc_fence_after();
    if (q < 2) {
        const uint32_t id = ptx::idesc_bf16(128, 64);
        const uint32_t c_d = q == 0 ? tm.ut : c_ot;
        const uint64_t bh = dsc(sm, q == 0 ? tl.nwh : tl.qeh), bl = dsc(sm, q == 0 ? tl.nwl : tl.qel);
#pragma unroll UNR
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t kb = ((ks >> 2) * BT64_KB + (ks & 3) * 32) >> 4;
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.sh + ks * 8, bh + kb, id, q == 0 || ks > 0);
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.sh + ks * 8, bl + kb, id, 1);
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.sl + ks * 8, bh + kb, id, 1);
        }
    }
    ptx::mma_commit(bar);
}

// fourth product: O^T += U^T P^T (issuer 0, all 64 chunk rows) and
// S^T += U^T (K o e^{G_C - G}) (issuer 1, all 128 key dims).
template <int UNR>
__device__ __forceinline__ void issue_fourth16(unsigned char* sm, uint32_t tmem, int q, const Bf16Tiles tl,
                                               const Bf16Tmem tm, uint32_t c_ot, uint64_t* bar)
{
    ptx::tc_fence_after();
    if (q < 2) {
        const uint32_t id = q == 0 ? ptx::idesc_bf16(128, 64) : ptx::idesc_bf16(128, 128);
        const uint32_t c_d = q == 0 ? c_ot : tm.st;
        const uint64_t bh = dsc(sm, q == 0 ? tl.ph : tl.kdh), bl = dsc(sm, q == 0 ? tl.pl : tl.kdl);
#pragma unroll UNR
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t kb = (ks * 32) >> 4;
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.uh + ks * 8, bh + kb, id, 1);
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.uh + ks * 8, bl + kb, id, 1);
            ptx::mma_bf16_ts(tmem + c_d, tmem + tm.ul + ks * 8, bh + kb, id, 1);
        }
    }
    ptx::mma_commit(bar);
}

// The products are issued by ISSUERS threads (lane 0 of warps 0..3, one per
// SM sub-partition), each owning a block of accumulator columns: a single
// issuing thread cannot keep the tensor core busy with these small (N <= 96)
// products.  Each accumulator still receives its MMAs in one thread's
// program order, so every element sums the same terms in the same order.
// All issuers commit to the same mbarrier (arrival count ISSUERS).
constexpr int ISSUERS = 4;
// Unrolling of the issue loops (4 by default).  Measured: full unrolling made
// the fused kernel slower (code size) and did not speed up the split chain,
// whose issue rate is set by the tensor pipe and by the other warps sharing
// the sub-partitions while it issues.
#ifndef KDA_ISSUE_UNROLL
#define KDA_ISSUE_UNROLL 4
#endif
#ifndef KDA_CHAIN_UNROLL
#define KDA_CHAIN_UNROLL 4
#endif
constexpr int ISSUE_UNROLL = KDA_ISSUE_UNROLL, CHAIN_UNROLL = KDA_CHAIN_UNROLL;
__device__ __forceinline__ int issuer(int tid) { return ((tid & 31) == 0 && tid < 32 * ISSUERS) ? tid >> 5 : -1; }

// first product.  Both operands come from shared memory, whose bandwidth bounds
// this product, so the A tile is not read twice by splitting N: issuer 0 runs
// D1, issuer 1 D1c, the others only commit.
template <int UNR>
__device__ __forceinline__ void issue_first(unsigned char* sm, uint32_t tmem, int q, uint64_t* bar)
{
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_tf32(128, 96);
    const uint64_t dbh = dsc(sm, SM_B1H);
    if (q == 0) {
        const uint64_t dak = dsc(sm, SM_AX + 8192), dbl = dsc(sm, SM_B1L);
#pragma unroll UNR
        for (int ks = 0; ks < 16; ++ks) {
            const uint32_t ka = ((ks >> 2) * AX_KB + (ks & 3) * 32) >> 4, kb = ((ks >> 2) * B1_KB + (ks & 3) * 32) >> 4;
            ptx::mma_tf32_ss(tmem + TM_D1, dak + ka, dbh + kb, id, ks > 0);
            ptx::mma_tf32_ss(tmem + TM_D1, dak + ka, dbl + kb, id, 1);
        }
    } else if (q == 1) {
        const uint64_t daq = dsc(sm, SM_AX);
#pragma unroll UNR
        for (int ks = 0; ks < 16; ++ks) {
            const uint32_t ka = ((ks >> 2) * AX_KB + (ks & 3) * 32) >> 4, kb = ((ks >> 2) * B1_KB + (ks & 3) * 32) >> 4;
            ptx::mma_tf32_ss(tmem + TM_D1C, daq + ka, dbh + kb, id, ks > 0);
        }
    }
    ptx::mma_commit(bar);
}

// second product.  Issuer q: W^T (q < 2) or U'^T (q >= 2), chunk rows [32 (q & 1), +32).
template <int UNR>
__device__ __forceinline__ void issue_second(unsigned char* sm, uint32_t tmem, int q, uint64_t* bar)
{
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_tf32(128, 32);
    const uint32_t hr = (q & 1) * 32, ho = (hr * 128) >> 4;
    const uint64_t dt = dsc(sm, SM_T) + ho;
#pragma unroll UNR
    for (int ks = 0; ks < 8; ++ks) {
        const uint64_t bd = dt + (((ks >> 2) * T64_KB + (ks & 3) * 32) >> 4);
        if (q < 2) {
            ptx::mma_tf32_ts(tmem + TM_WT + hr, tmem + TM_XT + ks * 8, bd, id, ks > 0);
        } else {
            ptx::mma_tf32_ts(tmem + TM_UT + hr, tmem + TM_YT + ks * 8, bd, id, ks > 0);
            ptx::mma_tf32_ts(tmem + TM_UT + hr, tmem + TM_YL + ks * 8, bd, id, 1);
        }
    }
    ptx::mma_commit(bar);
}

// The state-independent part of one chunk (all 512 threads): from the staged
// raw rows (q, k, v with the HALO rows before the chunk, gate f) and beta in
// shared memory, compute conv + SiLU, the gates and G, the first product (A
// and P), the solve for T and the second product.  On return (true) the
// tensor memory holds W^T and U'^T, shared memory the T, P (high, low),
// Q o e^G (high, low) and K o e^{G_C - G} (high, low) tiles, and ms.gamma
// holds e^{G_C}.  False: a tensor-core wait ran out (ms.err set).
struct ThreadConst {
    float wq[4], wk[4], wv[4];  // conv taps of this thread's q, k, v channel (4-tap form)
    float dtc, ea;              // dt_bias of this key dim, exp(A_log) of the head
};

__device__ __forceinline__ ThreadConst thread_const(const ChunkArgs& a, int h, int col)
{
    ThreadConst t;
    const int H = a.H, K = a.K;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int src = j - (4 - K);  // K < 4: the oldest taps are zero
        t.wq[j] = src >= 0 ? a.conv_w[((size_t)0 * H * D + h * D + col) * K + src] : 0.f;
        t.wk[j] = src >= 0 ? a.conv_w[((size_t)1 * H * D + h * D + col) * K + src] : 0.f;
        t.wv[j] = src >= 0 ? a.conv_w[((size_t)2 * H * D + h * D + col) * K + src] : 0.f;
    }
    t.dtc = a.dt_bias[(size_t)h * D + col];
    t.ea = expf(a.A_log[h]);
    return t;
}

// The chunk path's softplus log-decay, -ea * softplus(f + dt), with
// softplus(x) = max(x, 0) + log1p(e^-|x|): log1p(y) for y = e^-|x| in (0, 1]
// by the fast logarithm of 1 + y (absolute error ~4e-7) and, below 2^-7, by
// y - y^2/2 + y^3/3 - y^4/4 (truncation below 3e-11).  The prep, the split
// path's producers and its chunk-boundary pass all call this one function,
// so their chunk boundaries agree.
__device__ __forceinline__ float chunk_softplus_decay(float ea, float f, float dt)
{
    // explicit roundings: the same bits at every call site
    const float x = __fadd_rn(f, dt);
    const float y = exp_sfu(-fabsf(x));
    float p = __fmaf_rn(-0.25f, y, 0.33333334f);
    p = __fmaf_rn(-y, p, 0.5f);
    p = __fmaf_rn(-y, p, 1.0f);
    const float l1p = y < 0.0078125f ? __fmul_rn(y, p) : __logf(__fadd_rn(1.0f, y));
    return __fmul_rn(-ea, __fadd_rn(fmaxf(x, 0.0f), l1p));
}

// Unbounded gates: the number of rows this chunk takes, at most nvalid: the
// longest prefix over which every key dim's running log-decay G stays within
// 80 of the reference row of each 32-row half, so that every factor
// e^{+-(G_r - G_m)} the chunk forms is finite (|G_r - G_m| < 88 would do).
// With G held at row n - 1 beyond a prefix of n rows, the spans to check at
// row j are G_0 - G_j for j <= 16, G_16 - G_j for j < 32, G_32 - G_j for
// j <= 48 and G_48 - G_j after: each half's reference splits it into two
// spans, of which row 16 (48) closes the first.  A single row always fits.
// Rows past the cut get G held at the last row here, and zero q, k (their
// inverse norms) and beta from the caller, so they add nothing, as rows past
// a segment's end do.  G is this thread's 16 rows (absolute within the chunk).
__device__ __forceinline__ int chunk_cut(Misc& ms, int nvalid, float (&G)[RPT])
{
    const int tid = threadIdx.x, col = tid & (D - 1), qq = tid >> 7;
    if (tid == 0) ms.ncut = C;
    if ((qq & 1) == 0) ms.ganc[qq >> 1][col] = G[0];  // rows 0 and 32
    __syncthreads();
    int bad = C;
#pragma unroll
    for (int r = RPT - 1; r >= 0; --r) {
        // the span's start: this quarter's first row, but for rows 16 and 48
        // the first row of the quarter before
        const float g0 = (r == 0 && (qq & 1)) ? ms.ganc[qq >> 1][col] : G[0];
        if (g0 - G[r] > 80.0f) bad = RPT * qq + r;
    }
    bad = __reduce_min_sync(0xffffffffu, bad);
    if ((tid & 31) == 0 && bad < C) atomicMin(&ms.ncut, bad);
    __syncthreads();
    const int n = min(nvalid, ms.ncut);
    if (n < nvalid) {  // block-uniform
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            if (RPT * qq + r == n - 1) ms.ganc[0][col] = G[r];
        __syncthreads();
        const float gl = ms.ganc[0][col];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            if (RPT * qq + r >= n) G[r] = gl;
    }
    return n;
}

// The state-independent prep of a chunk: conv + SiLU, the gate and the running
// log-decay G of this thread's column and 16 rows, the q/k row norms applied.
// Registers and the prep scratch of ms only (e^{G_C} is stored by chunk_rest).
// UNB: either gate formula (the gates whose log-decays are not bounded by -5:
// softplus, or a lower bound below -5).  Returns the number of rows the chunk
// takes: nvalid, or with CUT possibly fewer (chunk_cut).
template <bool UNB, bool CUT = UNB>
__device__ __forceinline__ int chunk_prep(unsigned char* sm, Misc& ms, const ChunkArgs& a, const ThreadConst& tc,
                                          int nvalid, float (&qv)[RPT], float (&kv)[RPT], float (&vv)[RPT],
                                          float (&G)[RPT], bool zero_v = false)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = tid & (D - 1);
    const int qq = tid >> 7;
    const int lq = warp & 3;
    const int r0 = RPT * qq;
    const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(sm + SM_RAW);
    const __nv_bfloat16* rawf = reinterpret_cast<const __nv_bfloat16*>(sm + SM_RAWF);
    const float* wq = tc.wq;
    const float* wk = tc.wk;
    const float* wv = tc.wv;
    const float dtc = tc.dtc, ea = tc.ea;
    // ---- prep: conv + SiLU, gate, running log-decay for this thread's column and 16 rows,
    // two rows at a time in packed f32x2 arithmetic
    {
        float xq[5], xk[5], xv[5];  // raw rows lr .. lr + 4 (lr + 3 is row r's own)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            xq[j] = __bfloat162float(raw[0 * RAWR * D + (r0 + j) * D + col]);
            xk[j] = __bfloat162float(raw[1 * RAWR * D + (r0 + j) * D + col]);
            xv[j] = __bfloat162float(raw[2 * RAWR * D + (r0 + j) * D + col]);
        }
        const float2 dt2 = make_float2(dtc, dtc), ea2 = make_float2(ea, ea), lb2 = make_float2(a.lb, a.lb);
        const float2 one2 = make_float2(1.0f, 1.0f);
        const bool sp = UNB && a.gate_mode != KDA_GATE_SAFE;
        // softplus decays first, into a scratch over the previous chunk's dead
        // (K o e^{G_C - G})^T tiles: fewer values live than inside the conv loop
        float* lsc = reinterpret_cast<float*>(sm + SM_KD);
        if (sp) {
#pragma unroll 4
            for (int r = 0; r < RPT; ++r)
                lsc[(r0 + r) * D + col] = chunk_softplus_decay(ea, __bfloat162float(rawf[(r0 + r) * D + col]), dtc);
        }
        float run = 0.0f;
#pragma unroll
        for (int r = 0; r < RPT; r += 2) {
            const int lr = r0 + r;
#pragma unroll
            for (int j = 3; j < 5; ++j) {
                xq[j] = __bfloat162float(raw[0 * RAWR * D + (lr + j) * D + col]);
                xk[j] = __bfloat162float(raw[1 * RAWR * D + (lr + j) * D + col]);
                xv[j] = __bfloat162float(raw[2 * RAWR * D + (lr + j) * D + col]);
            }
            float2 aq = make_float2(0.f, 0.f), ak = aq, av = aq;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                aq = __ffma2_rn(make_float2(wq[j], wq[j]), make_float2(xq[j], xq[j + 1]), aq);
                ak = __ffma2_rn(make_float2(wk[j], wk[j]), make_float2(xk[j], xk[j + 1]), ak);
                av = __ffma2_rn(make_float2(wv[j], wv[j]), make_float2(xv[j], xv[j + 1]), av);
            }
            // SiLU: x / (1 + e^-x); the gate: lb * sigmoid(ea (f + dt))
            const float2 dq = __fadd2_rn(one2, make_float2(exp_sfu(-aq.x), exp_sfu(-aq.y)));
            const float2 dk = __fadd2_rn(one2, make_float2(exp_sfu(-ak.x), exp_sfu(-ak.y)));
            const float2 dv = __fadd2_rn(one2, make_float2(exp_sfu(-av.x), exp_sfu(-av.y)));
            const float2 sq = __fmul2_rn(aq, make_float2(rcp_sfu(dq.x), rcp_sfu(dq.y)));
            const float2 sk = __fmul2_rn(ak, make_float2(rcp_sfu(dk.x), rcp_sfu(dk.y)));
            const float2 sv = __fmul2_rn(av, make_float2(rcp_sfu(dv.x), rcp_sfu(dv.y)));
            float2 la;
            if (!sp) {
                const float f0 = __bfloat162float(rawf[lr * D + col]), f1 = __bfloat162float(rawf[(lr + 1) * D + col]);
                const float2 fz = __fmul2_rn(ea2, __fadd2_rn(make_float2(f0, f1), dt2));
                const float2 gd = __fadd2_rn(one2, make_float2(exp_sfu(-fz.x), exp_sfu(-fz.y)));
                la = __fmul2_rn(lb2, make_float2(rcp_sfu(gd.x), rcp_sfu(gd.y)));
            } else {
                la = make_float2(lsc[lr * D + col], lsc[(lr + 1) * D + col]);
            }
            const bool ok0 = lr < nvalid, ok1 = lr + 1 < nvalid;
            qv[r] = ok0 ? sq.x : 0.0f;
            kv[r] = ok0 ? sk.x : 0.0f;
            vv[r] = (ok0 && !zero_v) ? sv.x : 0.0f;  // a transfer run: zero values, so U' = 0
            qv[r + 1] = ok1 ? sq.y : 0.0f;
            kv[r + 1] = ok1 ? sk.y : 0.0f;
            vv[r + 1] = (ok1 && !zero_v) ? sv.y : 0.0f;
            run += ok0 ? la.x : 0.0f;
            G[r] = run;
            run += ok1 ? la.y : 0.0f;
            G[r + 1] = run;
#pragma unroll
            for (int j = 0; j < 3; ++j) { xq[j] = xq[j + 2]; xk[j] = xk[j + 2]; xv[j] = xv[j + 2]; }
        }
    }
    // row norms of q' and k' (this warp's 32 columns) and this quarter's log-decay total
    {
        float t[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) t[r] = qv[r] * qv[r];
        const float pq = transpose_reduce16(t, lane);
#pragma unroll
        for (int r = 0; r < RPT; ++r) t[r] = kv[r] * kv[r];
        const float pk = transpose_reduce16(t, lane);
        if (lane < 16) {
            ms.npart[0][qq][lq][lane] = pq;
            ms.npart[1][qq][lq][lane] = pk;
        }
        ms.gq[qq][col] = G[RPT - 1];
    }
    __syncthreads();
    int n = nvalid;
    {
        float off = 0.0f;
        for (int q2 = 0; q2 < qq; ++q2) off += ms.gq[q2][col];
#pragma unroll
        for (int r = 0; r < RPT; ++r) G[r] += off;
        if (CUT) n = chunk_cut(ms, nvalid, G);
        if (qq == 1) ms.gx[0][col] = G[0];          // row 16
        if (qq == 3) {
            ms.gx[1][col] = G[0];                   // row 48
            ms.gx[2][col] = G[RPT - 1];             // row 63 (G_C)
        }
    }
    if (tid < 2 * C) {
        const int qk = tid / C, r = tid % C;
        const float tot = ms.npart[qk][r >> 4][0][r & 15] + ms.npart[qk][r >> 4][1][r & 15] +
                          ms.npart[qk][r >> 4][2][r & 15] + ms.npart[qk][r >> 4][3][r & 15];
        // rows past a cut: zero q and k (and, below, beta: no update from v)
        ms.nrm[qk][r] = (!CUT || r < n) ? rsqrtf(tot + a.l2_eps) : 0.0f;
        if (CUT && qk == 0 && r >= n) ms.beta[r] = 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        qv[r] *= ms.nrm[0][r0 + r];
        kv[r] *= ms.nrm[1][r0 + r];
    }
    return n;
}

// The rest of the state-independent part of a chunk, from the prep's
// results: e^{G_C}, the operands, the first product, A and P, the solve for T
// and the second product (after chunk_prep: together the state-independent
// part of a chunk).  On return (true) the tensor memory holds W^T and U'^T,
// shared memory the T tile and the bf16 high/low P, Q o e^G and
// (K o e^{G_C - G})^T tiles, and ms.gamma holds e^{G_C}.  False: a
// tensor-core wait ran out (ms.err set).
struct NoHook {
    __device__ __forceinline__ void operator()() const {}
};

// hook(): run by every thread while the first product runs (the split
// producers' look-ahead for their next task; nothing in the fused kernel)
template <typename Hook = NoHook>
__device__ __forceinline__ bool chunk_rest(unsigned char* sm, Misc& ms, const ChunkArgs& a, int nvalid, uint32_t tmem,
                                           uint32_t lane_base, uint32_t& ph, float (&qv)[RPT], float (&kv)[RPT],
                                           float (&vv)[RPT], float (&G)[RPT], const Hook& hook = Hook())
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = tid & (D - 1);
    const int qq = tid >> 7;
    const int half = qq >> 1;
    const int lq = warp & 3;
    const int r0 = RPT * qq;
    (void)lq;
    if (qq == 3) ms.gamma[col] = exp_sfu(G[RPT - 1]);  // e^{G_C}; read after later block barriers
    // ---- operands of the first and second products; q^ e^G and k^ e^{G_C - G}
    // are formed here too and kept in registers until their tiles are free
    const float Gm = ms.gx[half][col];   // reference row 16 (first half) or 48 (second half)
    float qe[RPT], kdx[RPT];
    {
        const float Gm1 = ms.gx[1][col];
        const float GC = ms.gx[2][col];
        // the cross block (keys of the first half seen from the second half's
        // reference) is written by the first half; the second half writes its
        // own diagonal value a second time instead, which keeps this loop free
        // of per-half code paths
        const float Gx = half == 0 ? Gm1 : Gm;
        const int xrow = half == 0 ? 64 : 0;
        const float eGm = exp_sfu(Gm);          // first half: e^{G_16} >= e^{-85}
        const float cGC = exp_sfu(GC - Gm);     // second half: e^{G_63 - G_48} >= e^{-75}
        float xt[RPT], yt[RPT], yl[RPT];
        // two rows at a time in packed f32x2 arithmetic; the exponentials, TF32
        // roundings and the stores (one address per element) stay per element
        const float2 eGm2 = make_float2(eGm, eGm), cGC2 = make_float2(cGC, cGC);
        const float2 mGm2 = make_float2(-Gm, -Gm);
        auto lo2 = [](float2 x) {  // low parts of both lanes: x - trunc(x), exact in fp32
            return __fadd2_rn(x, make_float2(-__uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u),
                                             -__uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u)));
        };
#pragma unroll
        for (int r = 0; r < RPT; r += 2) {
            const int rr = r0 + r;
            const float2 dg = __fadd2_rn(make_float2(G[r], G[r + 1]), mGm2);  // G - Gm
            const float2 e = make_float2(exp_sfu(dg.x), exp_sfu(dg.y));
            const float2 ie = make_float2(exp_sfu(-dg.x), exp_sfu(-dg.y));
            const float2 k2 = make_float2(kv[r], kv[r + 1]), q2 = make_float2(qv[r], qv[r + 1]);
            const float2 ke = __fmul2_rn(k2, e), qe2 = __fmul2_rn(q2, e), kie = __fmul2_rn(k2, ie);
            const float2 qel = lo2(qe2), kiel = lo2(kie);
            const uint32_t o0 = swz(rr, col, AX_KB), o1 = swz(rr + 1, col, AX_KB);
            const uint32_t p0 = swz(rr, col, B1_KB), p1 = swz(rr + 1, col, B1_KB);
            st_hi(sm, SM_AX + 8192 + o0, ke.x);
            st_hi(sm, SM_AX + 8192 + o1, ke.y);
            st_raw(sm, SM_AX + 16384 + o0, qe2.x);
            st_raw(sm, SM_AX + 16384 + o1, qe2.y);
            st_raw(sm, SM_AX + o0, qel.x);
            st_raw(sm, SM_AX + o1, qel.y);
            st_raw(sm, SM_B1H + p0, kie.x);
            st_raw(sm, SM_B1H + p1, kie.y);
            st_raw(sm, SM_B1L + p0, kiel.x);
            st_raw(sm, SM_B1L + p1, kiel.y);
            // e^{G_r}: a product of two in-range factors in the first half; direct in the
            // second (e^{G_48} may underflow).  e^{G_C - G_r}: direct in the first half
            // (e^{G_C - G_16} may underflow); a product in the second.  The cross
            // factor is e^{G_48 - G_r} in the first half and e^{G_48 - G_r} = ie in
            // the second.  (half is uniform over a warp: one side runs.)
            float2 cross, eG, edec;
            if (half == 0) {
                cross = make_float2(exp_sfu(Gx - G[r]), exp_sfu(Gx - G[r + 1]));
                eG = __fmul2_rn(e, eGm2);
                edec = make_float2(exp_sfu(GC - G[r]), exp_sfu(GC - G[r + 1]));
            } else {
                cross = ie;
                eG = make_float2(exp_sfu(G[r]), exp_sfu(G[r + 1]));
                edec = __fmul2_rn(ie, cGC2);
            }
            const float2 kc = __fmul2_rn(k2, cross), kcl = lo2(kc);
            const uint32_t x0 = swz(xrow + rr, col, B1_KB), x1 = swz(xrow + rr + 1, col, B1_KB);
            st_raw(sm, SM_B1H + x0, kc.x);
            st_raw(sm, SM_B1H + x1, kc.y);
            st_raw(sm, SM_B1L + x0, kcl.x);
            st_raw(sm, SM_B1L + x1, kcl.y);
            const float2 qg = __fmul2_rn(q2, eG), kd2 = __fmul2_rn(k2, edec);
            qe[r] = qg.x;
            qe[r + 1] = qg.y;
            kdx[r] = kd2.x;
            kdx[r + 1] = kd2.y;
            const float2 be = make_float2(ms.beta[rr], ms.beta[rr + 1]);
            const float2 xg = __fmul2_rn(__fmul2_rn(be, k2), eG);
            xt[r] = tf32r(xg.x);
            xt[r + 1] = tf32r(xg.y);
            const float2 y = __fmul2_rn(be, make_float2(vv[r], vv[r + 1]));
            const float2 yl2 = lo2(y);
            yt[r] = y.x;
            yt[r + 1] = y.y;
            yl[r] = yl2.x;
            yl[r + 1] = yl2.y;
        }
        ptx::tmem_st16(tmem + lane_base + TM_XT + RPT * qq, xt);
        ptx::tmem_st16(tmem + lane_base + TM_YT + RPT * qq, yt);
        ptx::tmem_st16(tmem + lane_base + TM_YL + RPT * qq, yl);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- first product: D1 = [K~; Q~hi](B1hi + B1lo)^T, D1c = [Q~lo; K~] B1hi^T
    if (issuer(tid) >= 0) issue_first<ISSUE_UNROLL>(sm, tmem, issuer(tid), &ms.bar);
    hook();
    if (!wait_mma(ms, ph, a.dev_status)) return false;

    // ---- A (D1 lanes 0..63) and the D1c part of P.  D1 column of (row r,
    // key row s): the first half reads its own block (column s), the second
    // half its own block (column s >= 32) and, for s < 32, the cross block
    // (column 64 + s).  Warp (lane quarter lq, column group qq) reads columns
    // [32 qq, +32) for key rows [sb, sb + 32): group 0 serves rows r < 32,
    // group 2 rows r >= 32 and group 1 all rows.
    const int sb = qq == 1 ? 32 : 0;
    const bool dact = qq == 1 || (qq == 0) == ((col & 63) < 32);
    if (lq < 2 && qq < 3 && dact) {
        float* akk = reinterpret_cast<float*>(sm + SM_AKK);
        float* ptmp = reinterpret_cast<float*>(sm + SM_PTMP);
        const int r = col;
        const float br = ms.beta[r];
        float v[32], w[32];
        ptx::tmem_ld32(tmem + lane_base + TM_D1 + 32 * qq, v);
        ptx::tmem_ld32(tmem + lane_base + TM_D1C + 32 * qq, w);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            akk[r * 65 + sb + x] = sb + x < r ? br * v[x] : 0.0f;
            ptmp[r * 65 + sb + x] = w[x];
        }
    }
    __syncthreads();
    // ---- P = D1 lanes 64..127 + PTMP, masked to s <= r, as high and low
    // tiles (16-byte stores: four consecutive key rows share a swizzle chunk)
    if (lq >= 2 && qq < 3 && dact) {
        const float* ptmp = reinterpret_cast<const float*>(sm + SM_PTMP);
        const int r = col - 64;
        float v[32];
        ptx::tmem_ld32(tmem + lane_base + TM_D1 + 32 * qq, v);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
            float pv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s2 = sb + 4 * c4 + u;
                pv[u] = s2 <= r ? v[4 * c4 + u] + ptmp[r * 65 + s2] : 0.0f;
            }
            uint2 hi, lo;
            bf16_split2(pv[0], pv[1], hi.x, lo.x);
            bf16_split2(pv[2], pv[3], hi.y, lo.y);
            const uint32_t o = swz16(r, sb + 4 * c4, BT64_KB);
            *reinterpret_cast<uint2*>(sm + FUSED_TILES.ph + o) = hi;
            *reinterpret_cast<uint2*>(sm + FUSED_TILES.pl + o) = lo;
        }
    }
    // ---- Q o e^G and (K o e^{G_C - G})^T as bf16 high and low tiles for the
    // third and fourth products
    {
#pragma unroll
        for (int r = 0; r < RPT; r += 2) {  // element (row r0 + r, key dim col)
            uint32_t hi, lo;
            bf16_split2(qe[r], qe[r + 1], hi, lo);
            const uint32_t o0 = swz16(r0 + r, col, BT64_KB), o1 = swz16(r0 + r + 1, col, BT64_KB);
            *reinterpret_cast<uint16_t*>(sm + FUSED_TILES.qeh + o0) = (uint16_t)(hi & 0xFFFFu);
            *reinterpret_cast<uint16_t*>(sm + FUSED_TILES.qeh + o1) = (uint16_t)(hi >> 16);
            *reinterpret_cast<uint16_t*>(sm + FUSED_TILES.qel + o0) = (uint16_t)(lo & 0xFFFFu);
            *reinterpret_cast<uint16_t*>(sm + FUSED_TILES.qel + o1) = (uint16_t)(lo >> 16);
        }
        // KD^T row col, chunk rows [16 qq, +16) along K
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint2 hi, lo;
            bf16_split2(kdx[4 * j], kdx[4 * j + 1], hi.x, lo.x);
            bf16_split2(kdx[4 * j + 2], kdx[4 * j + 3], hi.y, lo.y);
            const uint32_t o = swz16(col, RPT * qq + 4 * j, BT128_KB);
            *reinterpret_cast<uint2*>(sm + FUSED_TILES.kdh + o) = hi;
            *reinterpret_cast<uint2*>(sm + FUSED_TILES.kdl + o) = lo;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();

    // ---- T = (I + A)^{-1} (unit lower triangular) in two levels.  The 32x32
    // diagonal halves are inverted by column-oriented forward substitution, one
    // row per lane and four columns per warp; the off-diagonal half follows as
    // T[H1,H0] = -inv(H1) A[H1,H0] inv(H0).  Each value goes to the fp32 copy
    // (operand of the later steps) and to the T operand tile as it is formed.
    {
        const float* akk = reinterpret_cast<const float*>(sm + SM_AKK);
        float* ts = reinterpret_cast<float*>(sm + SM_TS);
        {
            const int hb = warp >> 3, cb = (warp & 7) * 4, rb = 32 * hb;
            float av[31];  // this lane's row of A inside the half, zero on and above the diagonal
#pragma unroll
            for (int j = 0; j < 31; ++j) av[j] = lane > j ? akk[(rb + lane) * 65 + rb + j] : 0.0f;
            float x[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) x[c] = lane == cb + c ? 1.0f : 0.0f;
            // x_j is final once the steps before j are done (steps j < c add
            // exact zeros to column c)
#pragma unroll
            for (int j = 0; j < 31; ++j) {
#pragma unroll
                for (int c = 0; c < 4; ++c) x[c] = __fmaf_rn(-av[j], __shfl_sync(0xffffffffu, x[c], j), x[c]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ts[(rb + lane) * 65 + rb + cb + c] = x[c];
                st_hi(sm, SM_T + swz(rb + lane, rb + cb + c, T64_KB), x[c]);
            }
            // the block above the diagonal, rows [0, 32) x columns [32, 64), is zero
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int e = tid + e2 * NT;
                st_raw(sm, SM_T + swz(e >> 5, 32 + (e & 31), T64_KB), 0.0f);
            }
        }
        __syncthreads();
        {   // X = A[H1,H0] inv(H0).  inv(H0) is stored with its zeros above the
            // diagonal, so column y may start at any z <= y: at y rounded down to 4.
            // Warp w takes columns w and 31 - w, lane = row of X.
            const int y0 = warp, y1 = 31 - warp;
            const float* arow = akk + (32 + lane) * 65;
            float s0 = 0.0f, s1 = 0.0f;
            for (int z4 = y0 & ~3; z4 < (y1 & ~3); z4 += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) s0 = __fmaf_rn(arow[z4 + u], ts[(z4 + u) * 65 + y0], s0);
            }
            for (int z4 = y1 & ~3; z4 < 32; z4 += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float az = arow[z4 + u];
                    s0 = __fmaf_rn(az, ts[(z4 + u) * 65 + y0], s0);
                    s1 = __fmaf_rn(az, ts[(z4 + u) * 65 + y1], s1);
                }
            }
            ms.X[lane][y0] = s0;
            ms.X[lane][y1] = s1;
        }
        __syncthreads();
        {   // T[H1,H0] = -inv(H1) X.  inv(H1) is stored with its zeros above the
            // diagonal, so row x may end at any z >= x: at x rounded up to 4.
            // Warp w takes rows w and 31 - w, lane = column.
            const int x0 = warp, x1 = 31 - warp;
            const float* t0 = ts + (32 + x0) * 65 + 32;
            const float* t1 = ts + (32 + x1) * 65 + 32;
            float s0 = 0.0f, s1 = 0.0f;
            for (int z4 = 0; z4 <= x0; z4 += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float xz = ms.X[z4 + u][lane];
                    s0 = __fmaf_rn(t0[z4 + u], xz, s0);
                    s1 = __fmaf_rn(t1[z4 + u], xz, s1);
                }
            }
            for (int z4 = (x0 | 3) + 1; z4 <= x1; z4 += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) s1 = __fmaf_rn(t1[z4 + u], ms.X[z4 + u][lane], s1);
            }
            st_hi(sm, SM_T + swz(32 + x0, lane, T64_KB), -s0);
            st_hi(sm, SM_T + swz(32 + x1, lane, T64_KB), -s1);
        }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- second product: W^T = X^T T^T, U'^T = (Y + Ylo)^T T^T
    if (issuer(tid) >= 0) issue_second<ISSUE_UNROLL>(sm, tmem, issuer(tid), &ms.bar);
    if (!wait_mma(ms, ph, a.dev_status)) return false;
    return true;
}


// ---- inter-chunk steps shared by the fused kernel and the chain role of the
// split kernel; `t*` arguments are TMEM addresses (this warp's lane quarter
// included), `o*` shared-memory tile offsets.

// the output gate of this thread's 16 rows (bf16 bits, two rows per register)
__device__ __forceinline__ void load_gate_bits(uint32_t (&gp)[RPT / 2], const ChunkArgs& a, int c0, int r0,
                                               int nvalid, int h, int col)
{
#pragma unroll
    for (int x = 0; x < RPT / 2; ++x) gp[x] = 0u;
    if (a.g != nullptr) {
        const unsigned short* gb = static_cast<const unsigned short*>(a.g);
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const int r = r0 + x;
            const uint32_t bits = r < nvalid ? gb[((size_t)(c0 + r) * a.H + h) * D + col] : 0u;
            gp[x >> 1] |= bits << (16 * (x & 1));
        }
    }
}



// Outputs of this thread's 16 rows (lane j = col), optional gated RMSNorm, in
// two parts.  Part A (all threads) reads O^T, applies the scale and, when
// gated, leaves each warp's partial sums of squares in ms.epart; the caller
// then syncs the block.  Part B needs no block barrier: lanes 0..15 of every
// warp form the inverse RMS of the quarter's 16 rows from the four partials
// (the same sum in the same order in every warp) and the warp reads them back.
__device__ __forceinline__ void outputs_a_regs(Misc& ms, const ChunkArgs& a, float (&o)[RPT]);
__device__ __forceinline__ void write_outputs_a(Misc& ms, const ChunkArgs& a, uint32_t t_ot, float (&o)[RPT])
{
    ptx::tmem_ld16(t_ot, o);
    outputs_a_regs(ms, a, o);
}

// part A on this thread's 16 rows of O already in registers
__device__ __forceinline__ void outputs_a_regs(Misc& ms, const ChunkArgs& a, float (&o)[RPT])
{
    const int tid = threadIdx.x, lane = tid & 31, lq = (tid >> 5) & 3, qq = tid >> 7;
    const float2 sc2 = make_float2(a.scale, a.scale);
#pragma unroll
    for (int x = 0; x < RPT; x += 2) {
        const float2 y = __fmul2_rn(make_float2(o[x], o[x + 1]), sc2);
        o[x] = y.x;
        o[x + 1] = y.y;
    }
    if (a.g != nullptr) {
        float t[RPT];
#pragma unroll
        for (int x = 0; x < RPT; x += 2) {
            const float2 y = __fmul2_rn(make_float2(o[x], o[x + 1]), make_float2(o[x], o[x + 1]));
            t[x] = y.x;
            t[x + 1] = y.y;
        }
        const float pr = transpose_reduce16(t, lane);
        if (lane < 16) ms.epart[qq][lq][lane] = pr;
    }
}

__device__ __forceinline__ void write_outputs_b(Misc& ms, const ChunkArgs& a, float (&o)[RPT],
                                                const uint32_t (&gp)[RPT / 2], int c0, int nvalid, int h, float nw,
                                                void* outp)
{
    const int tid = threadIdx.x, lane = tid & 31, qq = tid >> 7, col = tid & (D - 1);
    const int r0 = RPT * qq, H = a.H;
    if (a.g != nullptr) {
        if (lane < 16) {
            const float tot = ms.epart[qq][0][lane] + ms.epart[qq][1][lane] + ms.epart[qq][2][lane] +
                              ms.epart[qq][3][lane];
            ms.rms[r0 + lane] = rsqrtf(tot * (1.0f / D) + a.norm_eps);  // same value from the quarter's 4 warps
        }
        __syncwarp();
        const float2 nw2 = make_float2(nw, nw);
#pragma unroll
        for (int x = 0; x < RPT; x += 2) {
            // o * rms * w * sigmoid(g), two rows per packed operation
            const float g0 = __uint_as_float(gp[x >> 1] << 16), g1 = __uint_as_float(gp[x >> 1] & 0xFFFF0000u);
            const float2 rr = *reinterpret_cast<const float2*>(&ms.rms[r0 + x]);
            const float2 y = __fmul2_rn(__fmul2_rn(make_float2(o[x], o[x + 1]), rr), nw2);
            const float2 z = __fmul2_rn(y, make_float2(sigmoidf_(g0), sigmoidf_(g1)));
            o[x] = z.x;
            o[x + 1] = z.y;
        }
    }
    if (a.out_bf16) {
        // bf16 pairs: lanes 2m and 2m+1 hold columns c and c+1; the even lane
        // stores rows [r0, r0+8) and the odd lane rows [r0+8, r0+16), both as
        // 4-byte (c, c+1) pairs, after one exchange per row
        const bool odd = lane & 1;
        const int cpair = col & ~1;
        __nv_bfloat162* ou = static_cast<__nv_bfloat162*>(outp);
#pragma unroll
        for (int x = 0; x < RPT / 2; ++x) {
            const float send = odd ? o[x] : o[RPT / 2 + x];
            const float got = __shfl_xor_sync(0xffffffffu, send, 1);
            const int r = r0 + (odd ? RPT / 2 : 0) + x;
            const float lo = odd ? got : o[x], hi = odd ? o[RPT / 2 + x] : got;
            if (r < nvalid) ou[(((size_t)(c0 + r) * H + h) * D + cpair) >> 1] = __floats2bfloat162_rn(lo, hi);
        }
    } else {
        const size_t ob = ((size_t)(c0 + r0) * H + h) * D + col;
        float* ou = static_cast<float*>(outp);
#pragma unroll
        for (int x = 0; x < RPT; ++x)
            if (r0 + x < nvalid) ou[ob + (size_t)x * H * D] = o[x];
    }
}

// A chunk starting `off` < HALO rows into its segment: the halo rows before
// the segment's first row are the carried conv state (oldest first; zero
// where K - 1 < HALO); the others were staged with the chunk.
__device__ __forceinline__ void patch_halo(unsigned char* sm, const ChunkArgs& a, int slot, int h, int off)
{
    const int H = a.H, K = a.K, conv_dim = 3 * H * D;
    const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(a.conv_state);
    __nv_bfloat16* rw = reinterpret_cast<__nv_bfloat16*>(sm + SM_RAW);
    for (int idx = threadIdx.x; idx < 3 * HALO * D; idx += NT) {
        const int tsel = idx / (HALO * D), sr = (idx / D) % HALO, cc = idx % D;
        const int x = off - HALO + sr;  // the halo row's position in the segment
        if (x >= 0) continue;
        const int cr = (K - 1) + x;
        rw[tsel * RAWR * D + sr * D + cc] =
            cr >= 0 ? cs[((size_t)slot * (K - 1) + cr) * conv_dim + (size_t)tsel * H * D + h * D + cc]
                    : __float2bfloat16_rn(0.0f);
    }
}

// wait (thread 0, bounded) for the raw-row copies of parity rph; all threads
// then observe the completed phase.  False: the wait ran out (ms.err set).
__device__ __forceinline__ bool wait_rows(Misc& ms, uint32_t& rph, int32_t* dev_status)
{
    if (threadIdx.x == 0 && !ptx::mbar_wait(&ms.rbar, rph)) {
        ms.err = 1;
        flag_status(dev_status, KDA_DEV_TIMEOUT);
    }
    __syncthreads();
    if (ms.err) return false;
    (void)ptx::mbar_try_wait(&ms.rbar, rph);  // completed: makes the copied rows visible to this thread
    rph ^= 1u;
    return true;
}

// SCAN: the instantiation for kda_prefill_scan, whose units past a.nsplit are
// transfer runs (zero values, outputs to a.out2); the others never test it.
template <bool UNB, bool SCAN = false>
__global__ void __launch_bounds__(NT, 1) kda_chunk_kernel(const ChunkArgs a, const __grid_constant__ RawMaps maps)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    Misc& ms = *reinterpret_cast<Misc*>(sm + SM_MISC);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int col = tid & (D - 1);  // channel / key dim / value dim / TMEM lane of this thread
    const int qq = tid >> 7;        // quarter: chunk rows [16 qq, 16 qq + 16); also the TMEM column group
    const int lq = warp & 3;        // TMEM lane quarter of this warp (lanes 32 lq ..)
    const int H = a.H, K = a.K;
    const int conv_dim = 3 * H * D;
    const int useq = a.schedule ? a.schedule[blockIdx.x / H] : blockIdx.x / H;  // the unit's sequence index
    const int h = blockIdx.x % H;
    const bool xfer = SCAN && a.nsplit > 0 && useq >= a.nsplit;  // a transfer run of the state scan
    const int seq = xfer ? useq - a.nsplit : useq;      // whose rows it reads

    // ---- unit checks (before any tensor-memory allocation)
    const int slot = a.slots ? a.slots[useq] : useq;
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

    const __nv_bfloat16* bg = static_cast<const __nv_bfloat16*>(a.b);
    __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state);

    if (tid == 0) {
        ptx::mbar_init(&ms.bar, ISSUERS);
        ptx::mbar_init(&ms.rbar, 1);
        ptx::fence_mbar_init();
        ms.err = 0;
        stage_chunk(sm, maps, ms, seg0, h);  // first chunk's rows, in flight during set-up
    }
    if (warp == 0) ptx::tmem_alloc(&ms.tmem, TM_COLS);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ms.tmem;
    const uint32_t lane_base = (uint32_t)(lq * 32) << 16;  // this warp's TMEM lane quarter
    uint32_t ph = 0;
    uint32_t rph = 0;        // parity of the raw-row copies being waited for
    bool rpending = true;    // raw-row copies issued and not yet waited for

    const ThreadConst tc = thread_const(a, h, col);
    const float nw = a.norm_w ? a.norm_w[col] : 1.0f;

    // ---- initial state -> TMEM S^T (lane j = col, key dims [32 qq, +32))
    {
        const float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = Sg[(size_t)(32 * qq + x) * D + col];
        ptx::tmem_st32(tmem + lane_base + TM_ST + 32 * qq, v);
    }

    // UNB (unbounded gates): chunks end where the decays leave the factored range
    // the new conv state: the sequence's last K-1 raw rows, from the staged rows
    // of the last chunk (nv valid rows)
    auto store_conv_state = [&](int nv) {
        const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(sm + SM_RAW);
        for (int idx = tid; idx < 3 * D * (K - 1); idx += NT) {
            const int r = idx / (3 * D), c = idx % (3 * D), tsel = c / D, cc = c % D;
            const int sr = HALO + nv - (K - 1) + r;
            cs[((size_t)slot * (K - 1) + r) * conv_dim + (size_t)tsel * H * D + h * D + cc] =
                raw[tsel * RAWR * D + sr * D + cc];
        }
    };
    float bnext = 0.0f;  // beta logit of row `tid` of the next chunk
    if (tid < C && seg0 + tid < seg1) bnext = __bfloat162float(bg[(size_t)(seg0 + tid) * H + h]);
    // A chunk's rows are staged as soon as the previous chunk's second product
    // has freed the staging region (two products and the outputs ahead of their use).
    for (int c0 = seg0; c0 < seg1 && !ms.err;) {
        const int nvalid = min(C, seg1 - c0);
        const int r0 = RPT * qq;

        if (tid < C) ms.beta[tid] = tid < nvalid ? sigmoidf_(bnext) : 0.0f;
        if (!wait_rows(ms, rph, a.dev_status)) break;
        rpending = false;
        if (c0 - seg0 < HALO) {
            // the rows before the segment are the conv state (only the first
            // chunk with fixed chunks; a short first chunk's successor too)
            patch_halo(sm, a, slot, h, c0 - seg0);
            __syncthreads();
        }
        if (!UNB && c0 + nvalid == seg1) store_conv_state(nvalid);
        int n;  // rows this chunk takes
        {
            float qv[RPT], kv[RPT], vv[RPT], G[RPT];
            n = chunk_prep<UNB>(sm, ms, a, tc, nvalid, qv, kv, vv, G, xfer);
            // the next chunk's beta logits: loaded now, used a chunk later
            if (tid < C && c0 + n + tid < seg1) bnext = __bfloat162float(bg[(size_t)(c0 + n + tid) * H + h]);
            if (UNB && c0 + n == seg1) {
                store_conv_state(n);  // the staged rows are still intact: read before the operands overwrite them
                __syncthreads();
            }
            if (!chunk_rest(sm, ms, a, n, tmem, lane_base, ph, qv, kv, vv, G)) break;
        }

        // the staging region is free: the next chunk's rows
        if (c0 + n < seg1) {
            if (tid == 0) stage_chunk(sm, maps, ms, c0 + n, h);
            rpending = true;
        }

        // ---- -W tile from W^T as bf16 high and low parts (lane i = col, rows [16 qq, +16));
        // S^T as bf16 high and low pairs (key dims [32 qq, +32))
        store_neg_w16(sm, FUSED_TILES, tmem + lane_base + TM_WT + RPT * qq, qq, col);
        state_split16(tmem + lane_base + TM_ST + 32 * qq, tmem + lane_base + TM_SH + 16 * qq,
                      tmem + lane_base + TM_SL16 + 16 * qq);
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();

        if (issuer(tid) >= 0)
            issue_third16<ISSUE_UNROLL>(sm, tmem, issuer(tid), FUSED_TILES, FUSED_TMEM, TM_OT, &ms.bar);
        if (!wait_mma(ms, ph, a.dev_status)) break;

        rescale_split16(tmem + lane_base + TM_ST + 32 * qq, tmem + lane_base + TM_UT + RPT * qq,
                        tmem + lane_base + TM_UH + 8 * qq, tmem + lane_base + TM_UL16 + 8 * qq, &ms.gamma[32 * qq]);
        ptx::tc_fence_before();
        __syncthreads();

        if (issuer(tid) >= 0)
            issue_fourth16<ISSUE_UNROLL>(sm, tmem, issuer(tid), FUSED_TILES, FUSED_TMEM, TM_OT, &ms.bar);
        uint32_t gp[RPT / 2];
        load_gate_bits(gp, a, c0, r0, n, h, col);  // while the product runs
        if (!wait_mma(ms, ph, a.dev_status)) break;

        {
            float o[RPT];
            write_outputs_a(ms, a, tmem + lane_base + TM_OT + RPT * qq, o);
            __syncthreads();
            write_outputs_b(ms, a, o, gp, c0, n, h, nw, xfer ? a.out2 : a.out);
        }
        ptx::tc_fence_before();
        __syncthreads();
        c0 += n;
    }

    // ---- final state S^T -> rec_state (S[i][j], lane j = col, key dims [32 qq, +32))
    // nothing may land in shared memory after the CTA ends
    if (tid == 0 && rpending) (void)ptx::mbar_wait(&ms.rbar, rph);
    if (!ms.err) {
        float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
        ptx::tmem_ld32(tmem + lane_base + TM_ST + 32 * qq, v);
#pragma unroll
        for (int x = 0; x < 32; ++x) Sg[(size_t)(32 * qq + x) * D + col] = v[x];
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------------
// Split prefill for few (sequence, head) chains (long prompts): one persistent
// cooperative grid, one CTA per SM.  CTA b < NC runs chain b: only the
// state-dependent products (third and fourth), chunk after chunk, leaving the
// raw outputs to kda_split_outputs_kernel (after the grid: the fused kernel's
// output steps).  The other CTAs are producers: they take (chain, chunk) tasks in
// chunk-major order, run the state-independent part of the chunk
// (chunk_prep and chunk_rest, the fused kernel's steps) and publish its operands -- -W,
// Q o e^G, P and (K o e^{G_C - G})^T as bf16 high and low tiles, U'^T and
// e^{G_C} in fp32 -- in a ring of SPLIT_RING slots per chain, with a release
// flag.  The chain waits for the flag, bulk-copies the tiles and returns the
// slot (a consumed counter the producer waits on before reusing it).  Both
// sides run the fused kernel's instructions on the same values (the producers
// publish the bf16 tiles chunk_rest builds; the chain runs the fused kernel's
// bf16 third and fourth products), so the results have the fused kernel's
// bits.  With unbounded gates the chunks are those of a chunk list fixed
// beforehand by the fused kernel's rule (kda_chunk_bounds_kernel), so the
// same holds.  All waits are bounded.

constexpr int SPLIT_RING = 8;
// Slot layout (bytes).  The chain's products run on bf16 operands split into a
// high and a low part (x = hi + lo to within 2^-16 |x|; three-term products
// hi*hi + hi*lo + lo*hi accumulate in fp32 at the bf16 tensor rate), in
// K-major 128-byte-swizzled tiles of 64 bf16 per row: third-product operands
// [0, 64 KiB) (-W and Q o e^G, 64 rows x 128 key dims), fourth-product
// operands [64 KiB, 112 KiB) (P, 64 x 64, and (K o e^{G_C - G})^T, 128 key
// dims x 64 rows), then U'^T and e^{G_C} in fp32.
constexpr uint32_t SL_NWH = 0, SL_NWL = 16384, SL_QEH = 32768, SL_QEL = 49152;
constexpr uint32_t SL_PH = 65536, SL_PL = 73728, SL_KDH = 81920, SL_KDL = 98304;
constexpr uint32_t SL_UT = 114688;   // U'^T: [quarter][lane][16] fp32
constexpr uint32_t SL_GAM = 147456;  // e^{G_C}: [128] fp32
constexpr uint32_t SLOT_BYTES = 147968;
constexpr uint32_t SL_A_BYTES = 65536, SL_B_BYTES = 49152;
// chain tile shared memory: the slot's first 112 KiB, same offsets.  Chain
// tensor memory: S^T (fp32), S^T high and low (bf16 pairs), U^T (fp32), U^T
// high and low (bf16 pairs), two O^T blocks (chunks alternate)
constexpr uint32_t CT_ST = 0, CT_SH = 128, CT_SL = 192, CT_UT = 256, CT_UH = 320, CT_UL = 352;
constexpr uint32_t CT_OT0 = 384, CT_OT1 = 448;
constexpr Bf16Tiles CHAIN_TILES{SL_NWH, SL_NWL, SL_QEH, SL_QEL, SL_PH, SL_PL, SL_KDH, SL_KDL};
constexpr Bf16Tmem CHAIN_TMEM{CT_ST, CT_SH, CT_SL, CT_UT, CT_UH, CT_UL};
static_assert(SL_A_BYTES + SL_B_BYTES <= (uint32_t)SM_MISC, "chain tiles overlap the scalars");
static_assert(SLOT_BYTES % 16 == 0 && SL_UT % 16 == 0 && SL_GAM % 16 == 0, "bulk copies need 16-byte pieces");

struct SplitArgs {
    int* ready;            // [NC][SPLIT_RING]: chunk index + 1 published in the slot
    int* consumed;         // [NC]: chunks the chain has finished reading
    unsigned char* ring;   // [NC][SPLIT_RING][SLOT_BYTES]
    int NC;                // chains = N * H
    // unbounded gates: chain u's chunks, bnd[u * bs] = count n, then the n
    // chunk starts and the segment's end (kda_chunk_bounds_kernel); null:
    // fixed 64-row chunks
    const int* bnd;
    int bs;
    uint32_t flag_polls;   // limit of every flag wait (polls with back-off)
    float* raw_o;          // [T][H][D]: the chains' outputs before scale, norm and gate
};

// chain u's number of chunks, and chunk c's first row and row count (UNB:
// from the chunk lists)
template <bool UNB>
__device__ __forceinline__ int split_nchunks(const SplitArgs& sp, int u, int seg0, int seg1)
{
    return UNB ? sp.bnd[(size_t)u * sp.bs] : (seg1 - seg0 + C - 1) / C;
}
template <bool UNB>
__device__ __forceinline__ void split_chunk(const SplitArgs& sp, int u, int c, int seg0, int seg1, int& c0, int& nv)
{
    if (UNB) {
        const int* b = sp.bnd + (size_t)u * sp.bs + 1;
        c0 = b[c];
        nv = b[c + 1] - c0;
    } else {
        c0 = seg0 + c * C;
        nv = min(C, seg1 - c0);
    }
}

__device__ __forceinline__ unsigned char* slot_ptr(const SplitArgs& sp, int u, int c)
{
    return sp.ring + ((size_t)u * SPLIT_RING + (c % SPLIT_RING)) * SLOT_BYTES;
}

// a chain unit's sequence range; false when the unit is skipped (and flagged)
__device__ __forceinline__ bool split_unit(const ChunkArgs& a, int u, int& slot, int& seg0, int& seg1, bool flag)
{
    const int seq = u / a.H;
    slot = a.slots ? a.slots[seq] : seq;
    if (slot < 0) return false;
    if (slot >= a.num_slots) {
        if (flag) flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
        return false;
    }
    seg0 = a.cu_seqlens[seq];
    seg1 = a.cu_seqlens[seq + 1];
    if (seg0 < 0 || seg1 < seg0 || seg1 > a.T) {
        if (flag) flag_status(a.dev_status, KDA_DEV_BAD_SEQLENS);
        return false;
    }
    return seg1 > seg0;
}

template <bool UNB>
__device__ void split_producer(unsigned char* sm, Misc& ms, const ChunkArgs& a, const RawMaps& maps,
                               const SplitArgs& sp, uint32_t tmem)
{
    const int tid = threadIdx.x, warp = tid >> 5, lq = warp & 3, qq = tid >> 7, col = tid & (D - 1);
    const uint32_t lane_base = (uint32_t)(lq * 32) << 16;
    const int H = a.H, NC = sp.NC;
    const int p = blockIdx.x - NC, NP = gridDim.x - NC;
    int maxc = 0;
    for (int u = 0; u < NC; u += (UNB ? 1 : H)) {  // fixed chunks: the same count for every head
        int slot, s0, s1;
        if (split_unit(a, u, slot, s0, s1, false)) maxc = max(maxc, split_nchunks<UNB>(sp, u, s0, s1));
    }
    uint32_t ph = 0, rph = 0;
    int cur_h = -1;
    ThreadConst tc;
    const __nv_bfloat16* bg = static_cast<const __nv_bfloat16*>(a.b);
    // The bulk copies that publish a task run on while the next task's rows
    // are staged and its prep runs (the staging region and the prep's
    // scratch lie below the published tiles).  Thread 0 waits for their
    // reads before the operand build overwrites the tiles and completes them
    // and releases the slot's flag while the first product runs -- or at
    // once, if the next task's slot is still taken (its chain may be waiting
    // for this very publication).
    int pend = -1;  // thread 0: the ready-flag index of a publication in flight, -1 none
    int pend_v = 0;
    auto complete_pending = [&]() {
        if (pend >= 0) {
            ptx::bulk_wait_all();
            ptx::fence_proxy_async_global();  // the bulk writes before the flag (release at gpu scope)
            ptx::st_release_gpu(&sp.ready[pend], pend_v);
            pend = -1;
        }
    };
    // A task's rows are staged as soon as the previous task's second product
    // has freed the staging region when that task is t + NP (the common case:
    // no skipped unit between them); the bookkeeping lives in shared memory.
    if (tid == 0) {
        ms.staged_t = -1;
        ms.rows_pending = 0;
        ms.next_ok = 0;
    }
    __syncthreads();
    for (int t = p; t < maxc * NC && !ms.err; t += NP) {
        const int c = t / NC, u = t % NC, h = u % H;
        int slot, seg0, seg1;
        if (!split_unit(a, u, slot, seg0, seg1, false)) continue;
        if (c >= split_nchunks<UNB>(sp, u, seg0, seg1)) continue;
        int c0, nvalid;
        split_chunk<UNB>(sp, u, c, seg0, seg1, c0, nvalid);
        if (h != cur_h) {
            tc = thread_const(a, h, col);
            cur_h = h;
        }
        const bool staged = ms.staged_t == t;
        if (tid == 0) {
            // the slot is free once the chain has read chunk c - SPLIT_RING (for a
            // staged task, checked while the previous task's first product ran)
            if (c >= SPLIT_RING && !(staged && ms.next_ok) &&
                ptx::ld_acquire_gpu(&sp.consumed[u]) < c - SPLIT_RING + 1) {
                complete_pending();
                if (!ptx::wait_flag_ge(&sp.consumed[u], c - SPLIT_RING + 1, sp.flag_polls)) {
                    ms.err = 1;
                    flag_status(a.dev_status, KDA_DEV_TIMEOUT);
                }
            }
            if (!ms.err && !staged) {
                stage_chunk(sm, maps, ms, c0, h);
                ms.rows_pending = 1;
            }
        }
        if (tid < C)
            ms.beta[tid] = staged ? ms.beta_next[tid]
                                  : (tid < nvalid ? sigmoidf_(__bfloat162float(bg[(size_t)(c0 + tid) * H + h])) : 0.0f);
        __syncthreads();
        if (ms.err) break;
        if (!wait_rows(ms, rph, a.dev_status)) break;
        if (tid == 0) ms.rows_pending = 0;
        if (c0 - seg0 < HALO) {
            patch_halo(sm, a, slot, h, c0 - seg0);
            __syncthreads();
        }
        float qv[RPT], kv[RPT], vv[RPT], G[RPT];
        if (UNB) {  // the softplus prep writes a scratch over a published tile: the copies must have read it
            if (tid == 0) complete_pending();
            __syncthreads();
        }
        chunk_prep<UNB, false>(sm, ms, a, tc, nvalid, qv, kv, vv, G);
        if (tid == 0 && pend >= 0) ptx::bulk_wait_read_all();  // released while the first product runs
        __syncthreads();  // the published tiles are read: the operand build may overwrite them
        // while the first product runs: the pending publication released, and
        // the next task's (t + NP) slot checked and beta loaded
        auto lookahead = [&]() {
            if (tid == 0) complete_pending();
            if (tid == 128 || (tid >= 256 && tid < 256 + C)) {
                const int tn = t + NP, cn = tn / NC, un = tn % NC;
                int sln, sn0, sn1, cn0, nvn;
                if (tn < maxc * NC && split_unit(a, un, sln, sn0, sn1, false) &&
                    cn < split_nchunks<UNB>(sp, un, sn0, sn1)) {
                    split_chunk<UNB>(sp, un, cn, sn0, sn1, cn0, nvn);
                    if (tid == 128) {
                        ms.next_ok = cn < SPLIT_RING || ptx::ld_acquire_gpu(&sp.consumed[un]) >= cn - SPLIT_RING + 1;
                    } else {
                        const int r = tid - 256;
                        ms.beta_next[r] =
                            r < nvn ? sigmoidf_(__bfloat162float(bg[(size_t)(cn0 + r) * H + un % H])) : 0.0f;
                    }
                }
            }
        };
        if (!chunk_rest(sm, ms, a, nvalid, tmem, lane_base, ph, qv, kv, vv, G, lookahead)) break;
        if (tid == 0) {  // the staging region is free: the next task's rows, if it is t + NP
            const int tn = t + NP, cn = tn / NC, un = tn % NC;
            int sln, sn0, sn1, cn0, nvn;
            if (tn < maxc * NC && split_unit(a, un, sln, sn0, sn1, false) &&
                cn < split_nchunks<UNB>(sp, un, sn0, sn1)) {
                split_chunk<UNB>(sp, un, cn, sn0, sn1, cn0, nvn);
                stage_chunk(sm, maps, ms, cn0, un % H);
                ms.staged_t = tn;
                ms.rows_pending = 1;
            }
        }

        // publish: the chain's operands as the bf16 high and low tiles
        // chunk_rest built (and -W from W^T), by bulk copies; U'^T and e^{G_C}
        // in fp32 by plain stores
        unsigned char* dst = slot_ptr(sp, u, c);
        store_neg_w16(sm, FUSED_TILES, tmem + lane_base + TM_WT + RPT * qq, qq, col);
        {
            float v[RPT];
            ptx::tmem_ld16(tmem + lane_base + TM_UT + RPT * qq, v);
            float4* ut = reinterpret_cast<float4*>(dst + SL_UT + ((size_t)qq * D + col) * RPT * 4);
#pragma unroll
            for (int j = 0; j < RPT / 4; ++j) ut[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            if (tid < D) reinterpret_cast<float*>(dst + SL_GAM)[tid] = ms.gamma[tid];
        }
        // no per-thread fence for these stores: the barrier orders them before
        // thread 0's fence and release of the flag (the grid-barrier pattern)
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::bulk_s2g(dst + SL_NWH, sm + FUSED_TILES.nwh, 32768);  // -W high, low
            ptx::bulk_s2g(dst + SL_QEH, sm + FUSED_TILES.qeh, 32768);  // Q o e^G high, low
            ptx::bulk_s2g(dst + SL_PH, sm + FUSED_TILES.ph, 16384);    // P high, low
            ptx::bulk_s2g(dst + SL_KDH, sm + FUSED_TILES.kdh, 32768);  // (K o e^{G_C - G})^T high, low
            ptx::bulk_commit();
            pend = u * SPLIT_RING + c % SPLIT_RING;  // completed and released during the next task
            pend_v = c + 1;
        }
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    }
    if (tid == 0) {
        complete_pending();  // the last publication (or one cut short by an error)
        // rows staged for a task that did not run (after an error) land before the CTA ends
        if (ms.rows_pending) (void)ptx::mbar_wait(&ms.rbar, rph);
    }
}

// bulk-copy one half of a published slot into the chain's tiles
__device__ __forceinline__ void chain_fetch(unsigned char* sm, uint64_t* bar, const unsigned char* src,
                                            uint32_t off, uint32_t bytes)
{
    ptx::mbar_arrive_expect_tx(bar, bytes);
    for (uint32_t o = 0; o < bytes; o += 32768)
        ptx::bulk_g2s(sm + off + o, src + off + o, min(32768u, bytes - o), bar);
}

template <bool UNB>
__device__ void split_chain(unsigned char* sm, Misc& ms, const ChunkArgs& a, const SplitArgs& sp, uint32_t tmem,
                            int u, int slot, int seg0, int seg1)
{
    const int tid = threadIdx.x, warp = tid >> 5, lq = warp & 3, qq = tid >> 7, col = tid & (D - 1);
    const uint32_t lane_base = (uint32_t)(lq * 32) << 16;
    const int H = a.H, K = a.K, h = u % H, r0 = RPT * qq;
    const int nchunks = split_nchunks<UNB>(sp, u, seg0, seg1);
    uint32_t ph = 0;
    bool pend_a = false, pend_b = false;

    {   // initial state -> TMEM S^T
        const float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = Sg[(size_t)(32 * qq + x) * D + col];
        ptx::tmem_st32(tmem + lane_base + CT_ST + 32 * qq, v);
    }

    // Wait (one thread, bounded, acquire) for chunk c's slot.  The block barrier
    // that follows every call orders the other threads' reads of the slot
    // after that acquire.  Thread 128 issues no products, so it can wait while
    // the issuers are busy.
    auto acquire_by = [&](int c, int who) {
        if (tid == who && !ptx::wait_flag_ge(&sp.ready[u * SPLIT_RING + c % SPLIT_RING], c + 1, sp.flag_polls)) {
            ms.err = 1;
            flag_status(a.dev_status, KDA_DEV_TIMEOUT);
        }
    };
    // U'^T (16 values of this thread) and e^{G_C} (tid < D) of chunk c, into registers
    float up[RPT], gam = 0.0f;
    auto load_ut = [&](int c) {
        const unsigned char* src = slot_ptr(sp, u, c);
        const float4* ut = reinterpret_cast<const float4*>(src + SL_UT + ((size_t)qq * D + col) * RPT * 4);
#pragma unroll
        for (int j = 0; j < RPT / 4; ++j) {
            const float4 x = ut[j];
            up[4 * j] = x.x; up[4 * j + 1] = x.y; up[4 * j + 2] = x.z; up[4 * j + 3] = x.w;
        }
        if (tid < D) gam = reinterpret_cast<const float*>(src + SL_GAM)[tid];
    };

    // The outputs of chunk c leave while the third product of chunk c + 1 runs
    // (O^T alternates between two TMEM column blocks), as they come from the
    // products: scale, gated norm and the final stores are the epilogue
    // kernel's, off the chain.  Chunk c + 1's slot is acquired and its U'^T
    // loaded during the third product too.
    auto store_raw = [&](uint32_t t_ot, int cc0, int cnv) {
        float o[RPT];
        ptx::tmem_ld16(t_ot, o);
        float* dst = sp.raw_o + ((size_t)(cc0 + r0) * H + h) * D + col;
#pragma unroll
        for (int x = 0; x < RPT; ++x)
            if (r0 + x < cnv) dst[(size_t)x * H * D] = o[x];
    };
    bool mma_pending = false;
    acquire_by(0, 0);
    __syncthreads();
    if (!ms.err) {
        if (tid == 0) {
            ptx::fence_proxy_async_global();
            chain_fetch(sm, &ms.rbar, slot_ptr(sp, u, 0), 0, SL_A_BYTES);
            chain_fetch(sm, &ms.bbar, slot_ptr(sp, u, 0), SL_A_BYTES, SL_B_BYTES);
        }
        pend_a = pend_b = true;
        load_ut(0);
    }
    int prev_c0 = 0, prev_nvalid = 0;
    bool have_prev = false;
    for (int c = 0; c < nchunks && !ms.err; ++c) {
        int c0, nvalid;
        split_chunk<UNB>(sp, u, c, seg0, seg1, c0, nvalid);
        const uint32_t c_ot = (c & 1) ? CT_OT1 : CT_OT0;
        ptx::tmem_st16(tmem + lane_base + CT_UT + RPT * qq, up);
        if (tid < D) ms.gamma[tid] = gam;
        state_split16(tmem + lane_base + CT_ST + 32 * qq, tmem + lane_base + CT_SH + 16 * qq,
                      tmem + lane_base + CT_SL + 16 * qq);
        if (tid == 0 && !ptx::mbar_wait(&ms.rbar, c & 1)) {
            ms.err = 1;
            flag_status(a.dev_status, KDA_DEV_TIMEOUT);
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (ms.err) break;
        pend_a = false;
        if (issuer(tid) >= 0) {
            (void)ptx::mbar_try_wait(&ms.rbar, c & 1);  // completed: the tiles are visible to this issuer
            issue_third16<CHAIN_UNROLL>(sm, tmem, issuer(tid), CHAIN_TILES, CHAIN_TMEM, c_ot, &ms.bar);
        }
        mma_pending = true;
        // while the third product runs: the previous chunk's O^T and norm
        // partials (the barrier of the wait below orders them before part B),
        // chunk c + 1's slot and U'^T
        if (have_prev) {
            store_raw(tmem + lane_base + (c_ot ^ (CT_OT0 ^ CT_OT1)) + RPT * qq, prev_c0, prev_nvalid);
            have_prev = false;
        }
        if (c + 1 < nchunks) acquire_by(c + 1, 128);
        __syncthreads();
        if (ms.err) break;
        if (c + 1 < nchunks) load_ut(c + 1);
        if (!wait_mma(ms, ph, a.dev_status)) break;
        mma_pending = false;

        // the third-product tiles are free: fetch chunk c + 1's
        if (c + 1 < nchunks) {
            if (tid == 0) {
                ptx::fence_proxy_async_global();
                chain_fetch(sm, &ms.rbar, slot_ptr(sp, u, c + 1), 0, SL_A_BYTES);
            }
            pend_a = true;
        }

        rescale_split16(tmem + lane_base + CT_ST + 32 * qq, tmem + lane_base + CT_UT + RPT * qq,
                        tmem + lane_base + CT_UH + 8 * qq, tmem + lane_base + CT_UL + 8 * qq, &ms.gamma[32 * qq]);
        if (tid == 0 && !ptx::mbar_wait(&ms.bbar, c & 1)) {
            ms.err = 1;
            flag_status(a.dev_status, KDA_DEV_TIMEOUT);
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (ms.err) break;
        pend_b = false;
        if (issuer(tid) >= 0) {
            (void)ptx::mbar_try_wait(&ms.bbar, c & 1);
            issue_fourth16<CHAIN_UNROLL>(sm, tmem, issuer(tid), CHAIN_TILES, CHAIN_TMEM, c_ot, &ms.bar);
        }
        mma_pending = true;
        // chunk c's slot is read (both tile copies have landed, U'^T and e^{G_C}
        // are in registers): hand it back (a thread that issues no products)
        if (tid == 128) ptx::st_release_gpu(&sp.consumed[u], c + 1);
        if (!wait_mma(ms, ph, a.dev_status)) break;
        mma_pending = false;

        // fetch chunk c + 1's fourth-product tiles
        if (tid == 0 && c + 1 < nchunks) chain_fetch(sm, &ms.bbar, slot_ptr(sp, u, c + 1), SL_A_BYTES, SL_B_BYTES);
        if (c + 1 < nchunks) pend_b = true;
        have_prev = true;
        prev_c0 = c0;
        prev_nvalid = nvalid;
    }
    if (have_prev && !ms.err) {
        const uint32_t c_ot = ((nchunks - 1) & 1) ? CT_OT1 : CT_OT0;
        store_raw(tmem + lane_base + c_ot + RPT * qq, prev_c0, prev_nvalid);
    }
    if (tid == 0 && mma_pending) (void)ptx::mbar_wait(&ms.bar, ph);  // after a failed wait: let the products end

    // nothing may land in shared memory after the CTA ends
    if (tid == 0) {
        if (pend_a) (void)ptx::mbar_wait(&ms.rbar, 0), (void)ptx::mbar_wait(&ms.rbar, 1);
        if (pend_b) (void)ptx::mbar_wait(&ms.bbar, 0), (void)ptx::mbar_wait(&ms.bbar, 1);
    }
    if (!ms.err) {
        float* Sg = a.rec_state + ((size_t)slot * H + h) * D * D;
        float v[32];
        ptx::tmem_ld32(tmem + lane_base + CT_ST + 32 * qq, v);
#pragma unroll
        for (int x = 0; x < 32; ++x) Sg[(size_t)(32 * qq + x) * D + col] = v[x];
        // the new conv state: the last K-1 raw rows of the sequence, older ones
        // from the carried state (each thread walks its channels' rows in order,
        // so a row is read before it is overwritten)
        const int len = seg1 - seg0, conv_dim = 3 * H * D;
        __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state);
        for (int c = tid; c < 3 * D; c += NT) {
            const int tsel = c / D, cc = c % D;
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(tsel == 0 ? a.q : (tsel == 1 ? a.k : a.v));
            for (int r = 0; r < K - 1; ++r) {
                const int sr = len - (K - 1) + r;  // row of the sequence, or < 0: carried row sr + K - 1
                const size_t ch = (size_t)tsel * H * D + h * D + cc;
                cs[((size_t)slot * (K - 1) + r) * conv_dim + ch] =
                    sr >= 0 ? src[((size_t)(seg0 + sr) * H + h) * D + cc]
                            : cs[((size_t)slot * (K - 1) + sr + K - 1) * conv_dim + ch];
            }
        }
    }
}

// The split path's output epilogue, after the split kernel: chunk c of
// chain blockIdx.y for c = blockIdx.x, + gridDim.x, ...; the fused kernel's
// output steps (scale, the gated RMSNorm with its per-warp partial sums in the
// same order, the stores) on the chains' raw outputs, with the same thread
// layout, so the results carry the fused kernel's bits.
template <bool UNB>
__global__ void __launch_bounds__(NT, 2) kda_split_outputs_kernel(const ChunkArgs a, const SplitArgs sp)
{
    __shared__ Misc ms;
    const int u = blockIdx.y, tid = threadIdx.x, qq = tid >> 7, col = tid & (D - 1), r0 = RPT * qq;
    int slot, seg0, seg1;
    if (!split_unit(a, u, slot, seg0, seg1, false)) return;
    const int H = a.H, h = u % H;
    const int nch = split_nchunks<UNB>(sp, u, seg0, seg1);
    const float nw = a.norm_w ? a.norm_w[col] : 1.0f;
    for (int c = blockIdx.x; c < nch; c += gridDim.x) {
        int c0, nvalid;
        split_chunk<UNB>(sp, u, c, seg0, seg1, c0, nvalid);
        // every load in flight at once: rows past the chunk's end read its last
        // row (in bounds) and are then zeroed
        float o[RPT];
        uint32_t gb16[RPT];
        const unsigned short* gbs = static_cast<const unsigned short*>(a.g);
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const int r = min(r0 + x, nvalid - 1);
            o[x] = sp.raw_o[((size_t)(c0 + r) * H + h) * D + col];
            gb16[x] = gbs ? gbs[((size_t)(c0 + r) * H + h) * D + col] : 0u;
        }
        uint32_t gp[RPT / 2];
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const bool ok = r0 + x < nvalid;
            o[x] = ok ? o[x] : 0.0f;
            if ((x & 1) == 0) gp[x >> 1] = 0u;
            gp[x >> 1] |= (ok ? gb16[x] : 0u) << (16 * (x & 1));
        }
        outputs_a_regs(ms, a, o);
        __syncthreads();
        write_outputs_b(ms, a, o, gp, c0, nvalid, h, nw, a.out);
        __syncthreads();  // the norm partials are reused by the next chunk
    }
}

template <bool UNB>
__global__ void __launch_bounds__(NT, 1)
    kda_chunk_split_kernel(const ChunkArgs a, const __grid_constant__ RawMaps maps, const SplitArgs sp)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    Misc& ms = *reinterpret_cast<Misc*>(sm + SM_MISC);
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool chain = (int)blockIdx.x < sp.NC;
    int slot = 0, seg0 = 0, seg1 = 0;
    if (chain && !split_unit(a, blockIdx.x, slot, seg0, seg1, tid == 0)) return;
    if ((ptx::smem_u32(sm) & 1023u) != 0) {
        if (tid == 0) flag_status(a.dev_status, KDA_DEV_TIMEOUT);
        return;
    }
    if (tid == 0) {
        ptx::mbar_init(&ms.bar, ISSUERS);
        ptx::mbar_init(&ms.rbar, 1);
        ptx::mbar_init(&ms.bbar, 1);
        ptx::fence_mbar_init();
        ms.err = 0;
    }
    if (warp == 0) ptx::tmem_alloc(&ms.tmem, TM_COLS);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ms.tmem;
    if (chain) split_chain<UNB>(sm, ms, a, sp, tmem, blockIdx.x, slot, seg0, seg1);
    else split_producer<UNB>(sm, ms, a, maps, sp, tmem);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, TM_COLS);
}

// Unbounded gates on the split path: each chain's chunk boundaries, fixed
// ahead of the producers by the fused kernel's own rule (chunk_cut) on the
// same running log-decays -- the gate in the prep's arithmetic, each
// quarter's sum in row order, then the quarter offsets -- so the chunks are
// the fused kernel's.  Chain u's list is bnd[u * bs]: the count n, the n
// chunk starts, the segment's end; bnd[u * bs + bs - 1] is the first 64-row
// chunk (from the segment's start) that gets cut.
//
// The rows of chunk [c0, c0 + nvalid) of (sequence seg, head h): returns the
// rows it takes (all threads).
__device__ __forceinline__ int bounds_chunk(Misc& ms, const ChunkArgs& a, int c0, int nvalid, int seg1, int h,
                                            float ea, float dtc)
{
    const int tid = threadIdx.x, col = tid & (D - 1), qq = tid >> 7, r0 = RPT * qq, H = a.H;
    const __nv_bfloat16* fg = static_cast<const __nv_bfloat16*>(a.f);
    float G[RPT];
    // all 16 rows' gates in flight at once (rows past the segment's end read
    // its last row, unused)
    __nv_bfloat16 fr[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) fr[r] = fg[((size_t)min(c0 + r0 + r, seg1 - 1) * H + h) * D + col];
    float run = 0.0f;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        float la = 0.0f;
        if (r0 + r < nvalid) {
            const float f = __bfloat162float(fr[r]);
            if (a.gate_mode == KDA_GATE_SAFE) {  // the prep's lb * sigmoid(ea (f + dt)), operation by operation
                const float fz = __fmul_rn(ea, __fadd_rn(f, dtc));
                la = __fmul_rn(a.lb, rcp_sfu(__fadd_rn(1.0f, exp_sfu(-fz))));
            } else {
                la = chunk_softplus_decay(ea, f, dtc);
            }
        }
        run += la;
        G[r] = run;
    }
    ms.gq[qq][col] = G[RPT - 1];
    __syncthreads();
    float off = 0.0f;
    for (int q2 = 0; q2 < qq; ++q2) off += ms.gq[q2][col];
#pragma unroll
    for (int r = 0; r < RPT; ++r) G[r] += off;
    return chunk_cut(ms, nvalid, G);
}

// Every 64-row chunk from a segment's start, in parallel (block = chunk
// blockIdx.x of chain blockIdx.y): the first one that gets cut, per chain.
// Up to there the chain's chunks are these; the list's last entry starts
// above any chunk index.
__global__ void __launch_bounds__(NT) kda_chunk_cutscan_kernel(const ChunkArgs a, int* bnd, int bs)
{
    __shared__ Misc ms;
    const int u = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, col = tid & (D - 1);
    int slot, seg0, seg1;
    if (!split_unit(a, u, slot, seg0, seg1, false)) return;
    const int c0 = seg0 + c * C;
    if (c0 >= seg1) return;
    const int h = u % a.H, nvalid = min(C, seg1 - c0);
    const int n = bounds_chunk(ms, a, c0, nvalid, seg1, h, expf(a.A_log[h]), a.dt_bias[(size_t)h * D + col]);
    if (tid == 0 && n < nvalid) atomicMin(bnd + (size_t)u * bs + bs - 1, c);
}

// The chunk lists: the 64-row chunks before each chain's first cut, then (one
// CTA per chain) its chunks one after another from there.
__global__ void __launch_bounds__(NT, 1) kda_chunk_bounds_kernel(const ChunkArgs a, int* bnd, int bs)
{
    __shared__ Misc ms;
    const int u = blockIdx.x, tid = threadIdx.x, col = tid & (D - 1);
    int* b = bnd + (size_t)u * bs;
    int slot, seg0, seg1;
    if (!split_unit(a, u, slot, seg0, seg1, false)) {
        if (tid == 0) b[0] = 0;
        return;
    }
    const int h = u % a.H;
    const int nfix = min(b[bs - 1], (seg1 - seg0 + C - 1) / C);  // whole 64-row chunks before the first cut
    for (int c = tid; c < nfix; c += NT) b[1 + c] = seg0 + c * C;
    int count = nfix;
    const float ea = expf(a.A_log[h]), dtc = a.dt_bias[(size_t)h * D + col];
    for (int c0 = seg0 + nfix * C; c0 < seg1;) {
        const int n = bounds_chunk(ms, a, c0, min(C, seg1 - c0), seg1, h, ea, dtc);
        if (tid == 0) b[1 + count] = c0;
        ++count;
        c0 += n;
    }
    if (tid == 0) {
        b[1 + count] = seg1;
        b[0] = count;
    }
}

}  // namespace chk

bool chunk_split_wanted(const kda_params* p, int N, int T)
{
    return chunk_supported(p) && (long long)N * p->num_heads <= 64 && T >= 1024;
}

size_t chunk_split_bytes(int N, int H)
{
    const size_t nc = (size_t)N * H;
    const size_t flags = (nc * (chk::SPLIT_RING + 1) * sizeof(int) + 1023) & ~size_t(1023);
    return flags + nc * chk::SPLIT_RING * chk::SLOT_BYTES;
}

bool chunk_supported(const kda_params* p)
{
    // dk = dv = 128 and bf16 rows, either gate
    return p->head_dim_k == 128 && p->head_dim_v == 128 && p->io_dtype == KDA_DTYPE_BF16;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [T][H * 128] bf16 rows (16-byte aligned base, row pitch H * 256 bytes); box of
// one head's 128 channels x box_rows rows; zero fill outside the tensor.
bool encode_rows(CUtensorMap* m, const void* base, int H, int T, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || base == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * chk::D, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * chk::D * 2};
    const cuuint32_t box[2] = {(cuuint32_t)chk::D, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk(int io_bf16, const ChunkArgs& a, cudaStream_t st)
{
    if (!io_bf16) return cudaErrorNotSupported;
    // per-row log decays bounded by -5 (safe gate, lb >= -5): fixed 64-row chunks
    const bool unb = !(a.gate_mode == KDA_GATE_SAFE && a.lb >= -5.0f);
    static PerDeviceOnce attr;
    cudaError_t ae = attr.run([](int) {
        const void* fns[4] = {(const void*)chk::kda_chunk_kernel<false>, (const void*)chk::kda_chunk_kernel<true>,
                              (const void*)chk::kda_chunk_kernel<false, true>,
                              (const void*)chk::kda_chunk_kernel<true, true>};
        cudaError_t e = cudaSuccess;
        for (int i = 0; i < 4 && e == cudaSuccess; ++i)
            e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, chk::SMEM_BYTES);
        return e;
    });
    if (ae != cudaSuccess) return ae;
    int dev = 0;
    cudaGetDevice(&dev);
    chk::RawMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (a.T > 0) {  // with no rows every unit returns before its first copy
        if (!encode_rows(&maps.q, a.q, a.H, a.T, chk::RAWR) || !encode_rows(&maps.k, a.k, a.H, a.T, chk::RAWR) ||
            !encode_rows(&maps.v, a.v, a.H, a.T, chk::RAWR) || !encode_rows(&maps.f, a.f, a.H, a.T, chk::C))
            return cudaErrorInvalidValue;
    }
    if (a.split_ws) {
        // split path: one cooperative grid of one CTA per SM, chains first
        static PerDeviceOnce split_attr;
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaError_t se = split_attr.run([](int) {
            cudaError_t e = cudaFuncSetAttribute(chk::kda_chunk_split_kernel<false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, chk::SMEM_BYTES);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(chk::kda_chunk_split_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, chk::SMEM_BYTES);
            return e;
        });
        if (se != cudaSuccess) return se;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chk::kda_chunk_split_kernel<false>, chk::NT,
                                                      chk::SMEM_BYTES);
        const int nc = a.N * a.H;
        if (per_sm >= 1 && 2 * nc <= sms) {
            chk::SplitArgs sp;
            const size_t flags = ((size_t)nc * (chk::SPLIT_RING + 1) * sizeof(int) + 1023) & ~size_t(1023);
            sp.ready = reinterpret_cast<int*>(a.split_ws);
            sp.consumed = sp.ready + (size_t)nc * chk::SPLIT_RING;
            sp.ring = a.split_ws + flags;
            sp.NC = nc;
            // unbounded gates: the chains' chunk lists after the ring
            int* bnd = unb ? reinterpret_cast<int*>(a.split_ws + chunk_split_bytes(a.N, a.H)) : nullptr;
            sp.bnd = bnd;
            sp.bs = a.T + 3;
            sp.flag_polls = a.dbg_chains_only_polls ? a.dbg_chains_only_polls : (1u << 25);
            sp.raw_o = reinterpret_cast<float*>(
                a.split_ws + chunk_split_bytes(a.N, a.H) +
                (unb ? (((size_t)nc * sp.bs * sizeof(int) + 1023) & ~size_t(1023)) : 0));
            cudaError_t e = cudaMemsetAsync(a.split_ws, 0, flags, st);
            if (e != cudaSuccess) return e;
            if (unb) {
                // first cut per chain: "none" (0x7f7f7f7f) until the scan finds one
                e = cudaMemsetAsync(bnd, 0x7f, (size_t)nc * sp.bs * sizeof(int), st);
                if (e != cudaSuccess) return e;
                chk::kda_chunk_cutscan_kernel<<<dim3((a.T + chk::C - 1) / chk::C, nc), chk::NT, 0, st>>>(a, bnd, sp.bs);
                chk::kda_chunk_bounds_kernel<<<nc, chk::NT, 0, st>>>(a, bnd, sp.bs);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
            ChunkArgs aa = a;
            void* args[] = {&aa, &maps, &sp};
            const void* fn = unb ? (const void*)chk::kda_chunk_split_kernel<true> : (const void*)chk::kda_chunk_split_kernel<false>;
            // test hook: the chains alone, so that their first flag wait runs out
            const int grid = a.dbg_chains_only_polls ? nc : sms;
            e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(chk::NT), args, chk::SMEM_BYTES, st);
            if (e != cudaSuccess || a.dbg_chains_only_polls) return e;
            // the output epilogue: four CTAs per SM's worth of CTAs over the chains' chunks (two resident)
            int gx = (4 * sms) / nc > 1 ? (4 * sms) / nc : 1;
            if (!unb && gx > (a.T + chk::C - 1) / chk::C) gx = (a.T + chk::C - 1) / chk::C;
            if (unb) chk::kda_split_outputs_kernel<true><<<dim3(gx, nc), chk::NT, 0, st>>>(a, sp);
            else chk::kda_split_outputs_kernel<false><<<dim3(gx, nc), chk::NT, 0, st>>>(a, sp);
            return cudaGetLastError();
        }
        // too few SMs for producers beside the chains: the fused kernel below
    }
    if (a.schedule) chk::kda_chunk_schedule_kernel<<<1, 256, 0, st>>>(a.cu_seqlens, a.N, a.nsplit, a.schedule);
    const dim3 grid(a.N * a.H);
    if (a.nsplit > 0) {  // kda_prefill_scan's zero-state and transfer runs
        if (unb) chk::kda_chunk_kernel<true, true><<<grid, chk::NT, chk::SMEM_BYTES, st>>>(a, maps);
        else chk::kda_chunk_kernel<false, true><<<grid, chk::NT, chk::SMEM_BYTES, st>>>(a, maps);
    } else if (unb) {
        chk::kda_chunk_kernel<true><<<grid, chk::NT, chk::SMEM_BYTES, st>>>(a, maps);
    } else {
        chk::kda_chunk_kernel<false><<<grid, chk::NT, chk::SMEM_BYTES, st>>>(a, maps);
    }
    return cudaGetLastError();
}

}  // namespace kda
