// kda_decode.cu -- decode at dk = dv = 128, the memory-bound serving step:
// a persistent kernel with one CTA on each of ~27/32 of the SMs, a producer
// warp that streams each unit's 64 KiB state, rows, conv history and
// parameters into a ring of shared-memory stages with bulk async copies, and
// 8 row warps that run the row (kda_row.cuh) on a loaded stage meanwhile and
// leave the new state in the stage, from where the producer stores it back
// with one bulk copy before reusing the stage.
#include "kda_row.cuh"

namespace kda {

// ------------------------------------------------------------------------
// Streaming decode (D = 128): persistent CTAs, producer warp + 8 consumer warps.
//
// CTA c owns a contiguous, head-major range of units (u = head * N + seq), so
// a CTA meets at most a couple of heads and loads each head's conv taps and
// dt_bias once.  The producer keeps DEC_STAGES units in flight.

// three stages fit in shared memory with bf16 rows, two with fp32 rows
template <typename IO> constexpr int dec_stages() { return sizeof(IO) == 2 ? 3 : 2; }

template <typename IO> struct DecStage {
    float S[DEC_D * DEC_D];        // the unit's state, row-major (64 KiB)
    IO rows[5][DEC_D];             // raw q, k, v, gate, output-gate rows
    IO hist[3][3][DEC_D];          // conv history [row][q|k|v][channel]
    float bval;                    // beta logit
    int slot;                      // state slot, or -1: skip the unit
    int head;                      // head of the unit (with slot: where the new state goes)
    int pad;
};

template <typename IO> struct DecSmem {
    static constexpr int STAGES = dec_stages<IO>();
    DecStage<IO> stage[STAGES];
    RowSmem<DEC_D> row;
    float normw[DEC_D];
    uint64_t full[STAGES], empty[STAGES];
};

template <typename IO>
__global__ void __launch_bounds__(DEC_THREADS, 1) kda_decode_stream_kernel(const RecArgs a)
{
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    DecSmem<IO>& sm = *reinterpret_cast<DecSmem<IO>*>(dyn_smem);
    constexpr int D = DEC_D;
    constexpr int DEC_STAGES = DecSmem<IO>::STAGES;
    constexpr int RPW = RecShape<D>::RPW, CPT = RecShape<D>::CPT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, K = a.K, N = a.N;
    const int conv_dim = H * 3 * D;
    const int units = N * H;
    const int u_begin = (int)(((long long)units * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);

    if (tid == 0) {
        for (int s = 0; s < DEC_STAGES; ++s) {
            ptx::mbar_init(&sm.full[s], 1);
            ptx::mbar_init(&sm.empty[s], REC_WARPS);  // one arrival per row warp
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();  // barrier initialisation visible to every thread
    // Programmatic dependent launch: the next kernel on the stream may start its
    // prologue now; every thread here waits for the previous kernel's completion
    // (and its memory) before its first global access.
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    // gain of column tid: read back only by the same thread (row_out)
    for (int c = tid; c < D; c += DEC_THREADS) sm.normw[c] = a.norm_w ? a.norm_w[c] : 1.0f;

    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const IO* f = static_cast<const IO*>(a.f);
    const IO* b = static_cast<const IO*>(a.b);
    const IO* g = static_cast<const IO*>(a.g);
    IO* cs = static_cast<IO*>(a.conv_state);
    const bool has_g = g != nullptr;

    if (warp == REC_WARPS) {
        // ---------------- producer: loads each unit into a stage and, once the
        // row warps have left the unit's new state in that stage, stores it back
        // with one bulk copy before the stage takes the next unit
        if (lane != 0) return;
        const uint64_t pol = ptx::policy_evict_first();
        // wait until the row warps are done with stage s (phase n) and write its state back
        auto write_back = [&](int s, int n) -> bool {
            if (!ptx::mbar_wait(&sm.empty[s], n & 1)) {
                flag_status(a.dev_status, KDA_DEV_TIMEOUT);
                return false;
            }
            DecStage<IO>& st = sm.stage[s];
            if (st.slot >= 0) {
                ptx::bulk_s2g(a.rec_state + ((size_t)st.slot * H + st.head) * D * D, st.S, D * D * 4);
                // the new conv state: the window's last K-1 raw rows (history rows 1.., then the current row)
                for (int r = 0; r < K - 1; ++r)
                    for (int seg = 0; seg < 3; ++seg)
                        ptx::bulk_s2g(cs + ((size_t)st.slot * (K - 1) + r) * conv_dim + (size_t)seg * H * D + st.head * D,
                                      r + 1 < K - 1 ? st.hist[r + 1][seg] : st.rows[seg], D * sizeof(IO));
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();  // the stage may be refilled
            }
            return true;
        };
        const int count = u_end - u_begin;
        for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
            const int s = i % DEC_STAGES, n = i / DEC_STAGES;
            if (n > 0 && !write_back(s, n - 1)) return;
            DecStage<IO>& st = sm.stage[s];
            const int h = u / N, seq = u % N;
            int slot = a.slots ? a.slots[seq] : seq;
            if (slot >= a.num_slots) {
                flag_status(a.dev_status, KDA_DEV_BAD_SLOT);
                slot = -1;
            }
            if (slot >= 0) {
                const uint32_t rowb = D * sizeof(IO);
                const uint32_t bytes = D * D * 4 + (has_g ? 5 : 4) * rowb + 3 * (K - 1) * rowb;
                asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(ptx::smem_u32(&sm.full[s])),
                             "r"(bytes) : "memory");
                ptx::bulk_g2s_stream(st.S, a.rec_state + ((size_t)slot * H + h) * D * D, D * D * 4, &sm.full[s], pol);
                const size_t rh = (size_t)seq * H + h;
                ptx::bulk_g2s(st.rows[0], q + rh * D, rowb, &sm.full[s]);
                ptx::bulk_g2s(st.rows[1], k + rh * D, rowb, &sm.full[s]);
                ptx::bulk_g2s(st.rows[2], v + rh * D, rowb, &sm.full[s]);
                ptx::bulk_g2s(st.rows[3], f + rh * D, rowb, &sm.full[s]);
                if (has_g) ptx::bulk_g2s(st.rows[4], g + rh * D, rowb, &sm.full[s]);
                for (int r = 0; r < K - 1; ++r)
                    for (int seg = 0; seg < 3; ++seg)
                        ptx::bulk_g2s(st.hist[r][seg],
                                      cs + ((size_t)slot * (K - 1) + r) * conv_dim + (size_t)seg * H * D + h * D,
                                      rowb, &sm.full[s]);
                st.bval = ldv(b + rh);
            }
            st.slot = slot;
            st.head = h;
            ptx::mbar_arrive(&sm.full[s]);
        }
        // the last units' states
        for (int i = count > DEC_STAGES ? count - DEC_STAGES : 0; i < count; ++i)
            if (!write_back(i % DEC_STAGES, i / DEC_STAGES)) return;
        ptx::bulk_wait_all();
        return;
    }

    // ---------------- consumers (256 threads)
    const int r0 = warp * RPW, c0 = lane * CPT;
    float sreg[RPW][CPT];
    int cur_head = -1;
    RowConst rc{a.gate_mode, a.lb, 0.0f, a.l2_eps, a.norm_eps, a.scale, sm.normw};
    for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
        const int s = i % DEC_STAGES, n = i / DEC_STAGES;
        const int h = u / N, seq = u % N;
        if (h != cur_head) {
            // this head's conv taps, dt_bias and decay scale (L2-resident), each
            // loaded by the thread whose row_conv item reads it: no barrier needed
            for (int it = tid; it < 4 * D; it += REC_THREADS) {
                if (it < 3 * D) {
                    const int ch = conv_channel<D>(it, h, H);
                    for (int j = 0; j < K; ++j) sm.row.cw[it][j] = a.conv_w[(size_t)ch * K + j];
                } else {
                    sm.row.dtb[it - 3 * D] = a.dt_bias[(size_t)h * D + it - 3 * D];
                }
            }
            rc.ea = expf(a.A_log[h]);
            cur_head = h;
        }
        if (!ptx::mbar_wait(&sm.full[s], n & 1)) {
            if (tid == 0) flag_status(a.dev_status, KDA_DEV_TIMEOUT);
            return;
        }
        DecStage<IO>& st = sm.stage[s];
        const int slot = st.slot;
        float bval = 0.0f, gval = 0.0f;
        if (slot < 0) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.empty[s]);  // nothing to write back
            continue;
        }
        load_tile_smem<D>(st.S, r0, c0, sreg);
        bval = st.bval;
        if (has_g && tid < D) gval = ldv(&st.rows[4][tid]);
        // the conv window straight from the stage: raw rows K-1 history rows, then the current row
        row_conv<D>(sm.row, K, rc,
                    [&](int c, int j) {
                        const int seg = c / D, ch = c % D;
                        return j < K - 1 ? ldv(&st.hist[j][seg][ch]) : ldv(&st.rows[seg][ch]);
                    },
                    [&](int i) { return ldv(&st.rows[3][i]); });
        row_delta<D>(sm.row, sreg, rc, bval);
        // the new state goes back into the stage (the producer stores it with one
        // bulk copy); the stores drain while the output step runs
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
            *reinterpret_cast<float4*>(st.S + (r0 + rr) * D + c0) =
                make_float4(sreg[rr][0], sreg[rr][1], sreg[rr][2], sreg[rr][3]);
        const float o = row_out<D>(sm.row, rc, gval, has_g);
        const size_t rh = (size_t)seq * H + h;
        if (tid < D) store_out(a.out, rh * D + tid, o, a.out_bf16);
        // Each warp hands its part of the stage back.  No block barrier: the next
        // unit's first writes to the row arrays come after its first barrier,
        // which every warp reaches only after the reads of this unit.
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.empty[s]);
    }
}

static_assert(sizeof(DecSmem<__nv_bfloat16>) <= 232448, "decode stage buffers exceed shared memory");
static_assert(sizeof(DecSmem<float>) <= 232448, "decode stage buffers exceed shared memory");

template <typename IO> static cudaError_t launch_decode_stream(const RecArgs& a, int units, cudaStream_t st)
{
    static PerDeviceOnce smem_attr;
    const int smem = (int)sizeof(DecSmem<IO>);
    cudaError_t e = smem_attr.run([&](int) {
        return cudaFuncSetAttribute(kda_decode_stream_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    // Streaming CTAs: about 27/32 of the SMs (128 of the 152 on GB300).  Measured:
    // more concurrent state streams lower the total HBM rate (B = 256 decode:
    // 6.24 TB/s with 128 CTAs, 5.86 TB/s with 152), while below ~112 CTAs the
    // per-SM stream rate (~50 GB/s) becomes the limit.
    const int cap = sm_count() * 27 / 32 > 0 ? sm_count() * 27 / 32 : 1;
    const int grid = units < cap ? units : cap;
    // launched as a programmatic dependent of the previous kernel on the stream:
    // the launch and the prologue overlap that kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_decode_stream_kernel<IO>, a);
}

cudaError_t launch_decode_stream_d128(int io_bf16, const RecArgs& a, int units, cudaStream_t st)
{
    return io_bf16 ? launch_decode_stream<__nv_bfloat16>(a, units, st) : launch_decode_stream<float>(a, units, st);
}

}  // namespace kda
