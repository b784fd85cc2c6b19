/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) layer.
 *
 * What the layer computes per (sequence, head), row by row (sources: ONNX
 * Runtime GenAI PR #2843 "Add BailingMoeV3 (Ling-3.0-tiny) KDA + MLA + MoE
 * model builder and CUDA plugin EP fallback", section "Summary of Changes";
 * TensorFold issue #850 "Ling-3.1-flash on CUDA: a shared KDA kernel
 * first...", comment of Oct 15):
 *   1. causal depthwise conv over the concatenated q|k|v channels with a
 *      carried conv state (the K-1 previous raw rows), then SiLU;
 *   2. q and k L2-normalised per head: x * (sum x^2 + l2_eps)^(-1/2);
 *   3. beta = sigmoid(b);
 *   4. per-key-dim log decay: softplus gate
 *          log alpha_i = -exp(A_log_h) * softplus(f_i + dt_bias_hi)
 *      or "safe" gate with lower bound lb < 0
 *          log alpha_i = lb * sigmoid(exp(A_log_h) * (f_i + dt_bias_hi));
 *   5. gated delta rule on the fp32 dk x dv state S (row i = key dim):
 *          S = (I - beta k k^T) Diag(alpha) S + beta k v^T ,  o = scale S^T q;
 *   6. optional sigmoid-gated RMSNorm over each head's dv outputs:
 *          y = o * (mean o^2 + norm_eps)^(-1/2) * w * sigmoid(g).
 *
 * Conventions for every call below:
 *   - All pointers except `p` (and the host-side params it holds) are DEVICE
 *     pointers, owned by the caller, 16-byte aligned, dense row-major.  The
 *     library allocates nothing, never synchronises the host, and only
 *     enqueues work on `stream`; calls are CUDA-graph capturable (see below).
 *   - Row tensors are token-major: q, k, gate f: [rows][H][dk]; v, out_gate g,
 *     out: [rows][H][dv]; beta logits b: [rows][H].  Row tensors and the conv
 *     state use p->io_dtype; `out` uses p->out_dtype.
 *   - Conv state: [num_slots][K-1][conv_dim], conv_dim = H*(2*dk+dv),
 *     channel order: all heads' q channels, then k, then v; oldest row first.
 *   - Recurrent state: fp32 [num_slots][H][dk][dv].
 *   - `slots` (nullable = identity) maps sequence b to its state slot; a
 *     negative slot skips the sequence entirely (no output, no state change).
 *   - States are updated in place; verify never writes them.  The conv
 *     state and the recurrent state are the whole hand-off between calls: a
 *     prompt prefilled and then decoded (or verified and committed) row by
 *     row continues one recurrence.  On the chunked prefill path with the
 *     safe gate and lb >= -5 a prompt cut into calls at multiples of 64 rows
 *     gives the bits of one uncut call (TensorFold #850, Oct 15 comment:
 *     chunks start at a segment's first row).  With a softplus gate or
 *     lb < -5 chunk boundaries follow the decays, so a cut call agrees with
 *     the uncut one to rounding, not bit for bit.
 *   - Under CUDA-graph capture a call keeps its pointers, sizes and params;
 *     the buffers' contents (rows, slot map, accepted counts) are read at
 *     each replay.  Make one call of each entry point on a device before
 *     capturing (it sets kernel attributes once).
 *   - `dev_status` (nullable): a device int32 into which kernels OR the
 *     KDA_DEV_* bits for input faults they detect (the faulty unit is
 *     skipped, never trapped).  The caller clears it.
 *   - Return value: KDA_OK, or a KDA_ERR_* code.  Argument, geometry and
 *     bound errors are returned before anything is launched (TensorFold
 *     #850, Oct 16 comment: reject unsupported KDA head widths and tap counts
 *     before launch; ORT #2843 review reply: validate the bound only in safe
 *     mode).  KDA_ERR_LAUNCH reports a failed launch.
 */
#ifndef KDA_GB300_KDA_H
#define KDA_GB300_KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Return codes. */
#define KDA_OK 0
#define KDA_ERR_INVALID_ARGUMENT 1     /* null / misaligned pointer, bad size or enum */
#define KDA_ERR_UNSUPPORTED_GEOMETRY 2 /* dk != dv, dk not in {32,64,128}, K not in {2,3,4} */
#define KDA_ERR_INVALID_BOUND 3        /* safe gate with lb not finite or >= 0 */
#define KDA_ERR_WORKSPACE 4            /* workspace missing or smaller than required */
#define KDA_ERR_LAUNCH 5               /* a kernel launch failed (cudaGetLastError) */
#define KDA_ERR_DEVICE 6               /* current device is not sm_103 */

/* Bits a kernel ORs into *dev_status. */
#define KDA_DEV_BAD_SEQLENS 1  /* cu_seqlens not monotone or outside [0, T] */
#define KDA_DEV_BAD_SLOT 2     /* slots[b] >= num_slots */
#define KDA_DEV_BAD_ACCEPTED 4 /* accepted[b] outside [0, W] */
#define KDA_DEV_TIMEOUT 8      /* a bounded on-chip wait gave up; the unit was skipped */

#define KDA_DTYPE_F32 0
#define KDA_DTYPE_BF16 1

#define KDA_GATE_SOFTPLUS 0
#define KDA_GATE_SAFE 1

/* Per-layer configuration, read on the host at each call.  The four
 * parameter pointers are device pointers. */
typedef struct kda_params {
    int32_t num_heads;        /* H >= 1                                        */
    int32_t head_dim_k;       /* dk in {32, 64, 128}                           */
    int32_t head_dim_v;       /* dv == dk                                      */
    int32_t conv_kernel;      /* K in {2, 3, 4}                                */
    int32_t gate_mode;        /* KDA_GATE_SOFTPLUS or KDA_GATE_SAFE            */
    float gate_lower_bound;   /* lb < 0, finite; read only in safe mode        */
    float l2_eps;             /* q/k L2-norm epsilon, >= 0 (1e-6)              */
    float norm_eps;           /* output RMSNorm epsilon, >= 0 (1e-6)           */
    float scale;              /* output scale, finite (1.0)                    */
    int32_t io_dtype;         /* rows and conv state: KDA_DTYPE_F32 / _BF16    */
    int32_t out_dtype;        /* out: KDA_DTYPE_F32 / _BF16                    */
    int32_t num_slots;        /* state slots in the conv / recurrent buffers   */
    const float* A_log;       /* [H] fp32                                      */
    const float* dt_bias;     /* [H][dk] fp32                                  */
    const float* conv_weight; /* [conv_dim][K] fp32, tap K-1 = current row     */
    const float* norm_weight; /* [dv] fp32, nullable = unit weight             */
} kda_params;

/*
 * Variable-length prefill ("prompt rows").  Sequence s owns rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of the row tensors; its chunks restart
 * at the segment's first row (TensorFold #850, Oct 15 comment: prompt rows in
 * chunks from a segment's first row; ORT #2843: VarlenCausalConvWithState).
 *   cu_seqlens: device int32 [N+1], cu_seqlens[0] = 0, monotone, last = T.
 *   out_gate:   nullable; when given the gated RMSNorm epilogue is applied.
 *   conv_state, rec_state: read as the initial states of each sequence and
 *               overwritten with the final ones.  A zero-length sequence
 *               leaves both unchanged.
 *   workspace:  device scratch of at least kda_prefill_workspace_bytes(p,N,T)
 *               bytes (may be NULL when that is 0); contents need no init.
 */
KDA_API int kda_prefill_varlen(const kda_params* p, const int32_t* cu_seqlens, int32_t N,
                               int32_t T, const void* q, const void* k, const void* v,
                               const void* gate, const void* beta, const void* out_gate,
                               const int32_t* slots, void* conv_state, float* rec_state,
                               void* out, void* workspace, size_t ws_bytes,
                               int32_t* dev_status, cudaStream_t stream);

/* Scratch bytes kda_prefill_varlen needs for N sequences and T rows: a few
 * bytes per sequence; for few long sequences (N * H <= 64, T >= 1024, the
 * producer / chain path) also the operand ring and T * H * dv fp32 values
 * for the chains' outputs before their gated norm. */
KDA_API size_t kda_prefill_workspace_bytes(const kda_params* p, int32_t N, int32_t T);

/*
 * kda_prefill_varlen without a caller-provided workspace, for callers that
 * cannot allocate device memory (an allocator-free runtime, a plugin barred
 * from the host's memory pools, a serving loop that must never call
 * cudaMalloc).  The source pages have no counterpart: this is a service of
 * this library.  Arguments and results are those of kda_prefill_varlen; the
 * scratch is a fixed array of kda_prefill_static_workspace_capacity() bytes
 * (256 KiB: up to 65535 sequences per call) in the library's device memory
 * on every GPU that uses it, kept until the process exits.
 *   - Allocates nothing and calls no allocating routine.
 *   - Returns KDA_ERR_WORKSPACE, before any launch, when N needs more scratch
 *     than the array holds.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress), and so does the first call after the device's
 *     context changed (cudaDeviceReset, a new primary context); make those
 *     calls before any stream capture.
 *   - All calls share the array.  Calls whose kernels could run at the same
 *     time on one GPU (unordered streams) race on it: order them.
 */
KDA_API int kda_prefill_varlen_static_ws(const kda_params* p, const int32_t* cu_seqlens, int32_t N,
                                         int32_t T, const void* q, const void* k, const void* v,
                                         const void* gate, const void* beta, const void* out_gate,
                                         const int32_t* slots, void* conv_state, float* rec_state,
                                         void* out, int32_t* dev_status, cudaStream_t stream);

/* Bytes of the built-in scratch behind kda_prefill_varlen_static_ws. */
KDA_API size_t kda_prefill_static_workspace_capacity(void);

/*
 * Chunk-parallel prefill by an affine state scan: the context-parallel form
 * of kda_prefill_varlen (same arguments and results, same supported shape as
 * its tensor-core path: bf16 rows, dk = dv = 128), for long sequences.  The
 * delta rule is linear in the state, so over any run of rows
 *     S_out = M S_in + N   and   o_r = obar_r + psi_r S_in,
 * with (N, obar) what the rows give from a zero state and (M, psi) what they
 * give from the identity with zero values.  Each sequence is cut into
 * `segments` pieces of whole 64-row chunks (TensorFold #850, Oct 15 comment:
 * chunks from a segment's first row); all pieces run at once (zero-state and
 * transfer runs, one launch of the chunk kernel); a scan S_{p+1} = M_p S_p +
 * N_p gives each piece's start state; a fix-up adds psi_r S_p to the outputs
 * and applies the gated RMSNorm.  On several GPUs each would take its own
 * pieces and only the states of the scan would travel; here the pieces share
 * one GPU.
 *   - Results agree with kda_prefill_varlen and the serial recurrence to
 *     rounding, not bit for bit (another summation order); prompt-cut bit
 *     identity does not hold across the two entry points.
 *   - workspace: kda_prefill_scan_workspace_bytes(p, N, T, segments) bytes,
 *     16-byte aligned (about 1 KiB per row-head: raw outputs and corrections
 *     in fp32, plus two states per piece and head).
 *   - segments in [1, KDA_SCAN_MAX_SEGMENTS]; other shapes of p give
 *     KDA_ERR_UNSUPPORTED_GEOMETRY, before any launch.
 */
#define KDA_SCAN_MAX_SEGMENTS 64
KDA_API int kda_prefill_scan(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T, const void* q,
                             const void* k, const void* v, const void* gate, const void* beta, const void* out_gate,
                             const int32_t* slots, void* conv_state, float* rec_state, void* out, void* workspace,
                             size_t ws_bytes, int32_t segments, int32_t* dev_status, cudaStream_t stream);

/* Workspace bytes of kda_prefill_scan (0 for an unsupported shape). */
KDA_API size_t kda_prefill_scan_workspace_bytes(const kda_params* p, int32_t N, int32_t T, int32_t segments);

/*
 * Test hook for the bounded on-chip waits (no counterpart on the source
 * pages).  Same arguments as kda_prefill_varlen for a long-prompt shape that
 * takes the split (producer / chain) path -- bf16 rows, dk = dv = 128, the safe
 * gate with lb >= -5, N * H <= 64, T >= 1024 -- plus a poll limit.  Launches
 * only the chain CTAs, without the producers that publish their operands, and
 * limits every flag wait to `poll_limit` polls (about a microsecond each):
 * each chain's first wait runs out, the chain sets KDA_DEV_TIMEOUT in
 * *dev_status and returns with nothing in flight, leaving the states and the
 * context as they were.  Returns KDA_ERR_INVALID_ARGUMENT for any other shape
 * or a zero limit.  The failure is made on the host (the producers are not
 * launched); nothing faults or traps.
 */
KDA_API int kda_debug_split_chains_only(const kda_params* p, const int32_t* cu_seqlens, int32_t N, int32_t T,
                                        const void* q, const void* k, const void* v, const void* gate,
                                        const void* beta, const void* out_gate, const int32_t* slots,
                                        void* conv_state, float* rec_state, void* out, void* workspace,
                                        size_t ws_bytes, int32_t* dev_status, uint32_t poll_limit,
                                        cudaStream_t stream);

/*
 * Test hook for the device activations every kernel shares (no counterpart
 * on the source pages; the pages name the functions, not their arithmetic):
 * y[i] = f(x[i]) for i < n, with f by `which`:
 *   KDA_ACT_EXP     e^x (on the special-function unit's base-2 exponential)
 *   KDA_ACT_RCP     1/x
 *   KDA_ACT_SIGMOID 1/(1 + e^-x)   (beta, the safe gate, the output gate)
 *   KDA_ACT_SILU    x/(1 + e^-x)   (after the causal conv)
 * x and y are device arrays of n floats (n >= 0; they may alias), 16-byte
 * aligned.  Returns KDA_ERR_INVALID_ARGUMENT for an unknown `which`, n < 0,
 * or (n > 0) a null or misaligned pointer, all before any launch;
 * KDA_ERR_LAUNCH if the launch fails.
 */
#define KDA_ACT_EXP 0
#define KDA_ACT_RCP 1
#define KDA_ACT_SIGMOID 2
#define KDA_ACT_SILU 3
KDA_API int kda_debug_activations(int32_t which, const float* x, float* y, int32_t n, cudaStream_t stream);

/*
 * Decode: one row per sequence, B sequences (row b belongs to sequence b).
 * Updates the conv and recurrent states in place and writes out [B][H][dv]
 * (TensorFold #850, Oct 15 comment: decode rows).
 */
KDA_API int kda_decode(const kda_params* p, int32_t B, const void* q, const void* k,
                       const void* v, const void* gate, const void* beta,
                       const void* out_gate, const int32_t* slots, void* conv_state,
                       float* rec_state, void* out, int32_t* dev_status,
                       cudaStream_t stream);

/*
 * Speculative verify window: W draft rows per sequence (rows b*W .. b*W+W-1),
 * run on read-only copies of the states.  Writes out [B*W][H][dv] -- each
 * row bit-identical to what serial kda_decode calls would produce -- and a
 * log of each row's decay, normalised key and update plus its raw conv row,
 * so that kda_commit can replay any accepted prefix exactly (TensorFold #850,
 * Oct 15 comment: a window logs each row's decay, normalized key and update;
 * SGLang PR #33561: fused conv + gating + recurrent verify).
 *   log: device scratch of kda_verify_log_bytes(p, B, W) bytes, written here
 *        and read by kda_commit; opaque layout.
 */
KDA_API int kda_verify_window(const kda_params* p, int32_t B, int32_t W, const void* q,
                              const void* k, const void* v, const void* gate,
                              const void* beta, const void* out_gate,
                              const int32_t* slots, const void* conv_state,
                              const float* rec_state, void* log, void* out,
                              int32_t* dev_status, cudaStream_t stream);

/* Bytes of the verify log for B sequences and W rows. */
KDA_API size_t kda_verify_log_bytes(const kda_params* p, int32_t B, int32_t W);

/*
 * Commit the accepted prefix of each sequence's last verify window: for
 * sequence b, replay rows 0 .. accepted[b]-1 from the log onto its states,
 * leaving them bit-identical to accepted[b] serial kda_decode calls
 * (SGLang PR #33561: KDA state commit after target-verify).  accepted[b] = 0
 * changes nothing.  `slots`, B and W must match the verify call.
 *   accepted: device int32 [B], each in [0, W].
 */
KDA_API int kda_commit(const kda_params* p, int32_t B, int32_t W, const int32_t* accepted,
                       const int32_t* slots, const void* log, void* conv_state,
                       float* rec_state, int32_t* dev_status, cudaStream_t stream);

/*
 * Commit and verify in one call: for each sequence b, first replay rows
 * 0 .. accepted[b]-1 of the PREVIOUS window from log_prev onto its states and
 * store the committed states (exactly what kda_commit does), then verify the
 * NEW window's W draft rows on the committed states (exactly what
 * kda_verify_window does), writing `out` and the new window's `log`.  The
 * results carry the bits of kda_commit followed by kda_verify_window; the
 * state is read once instead of twice (TensorFold #850, Oct 15 comment: the
 * next window first replays the kept rows of the last one).
 *   accepted: device int32 [B], rows of the previous window to keep, each in
 *             [0, W]; a sequence with an out-of-range count is flagged
 *             (KDA_DEV_BAD_ACCEPTED) and skipped entirely (no commit, no
 *             outputs, no log rows).
 *   log_prev: the previous window's log (kda_verify_window or
 *             kda_commit_verify with the same p, B, W and slots); read only.
 *   log:      this window's log, kda_verify_log_bytes(p, B, W) bytes; may be
 *             the same buffer as log_prev (each sequence's rows are read
 *             before they are rewritten).
 * Other arguments as in kda_verify_window; conv_state and rec_state are
 * updated in place by the commit.
 */
KDA_API int kda_commit_verify(const kda_params* p, int32_t B, int32_t W, const int32_t* accepted,
                              const void* log_prev, const void* q, const void* k, const void* v,
                              const void* gate, const void* beta, const void* out_gate,
                              const int32_t* slots, void* conv_state, float* rec_state, void* log,
                              void* out, int32_t* dev_status, cudaStream_t stream);

/* Human-readable name of a return code. */
KDA_API const char* kda_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
KDA_API int kda_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_GB300_KDA_H */
