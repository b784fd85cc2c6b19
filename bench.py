"""KDA layer throughput on GB300: tokens/s and fraction of the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|verify|prefill_varlen|prefill_long|...] [--no-legs]

With --gpus N > 1 outside torchrun the script relaunches itself under
torch.distributed.run with N processes (one per GPU).

One step is one pass of the layer's hot path over one batch of seeded
synthetic input.  The headline workload is the decode step (64 sequences x
1 row, 32 heads, dk = dv = 128, bf16 rows, fp32 state, softplus gate, gated
RMSNorm epilogue): one kda_decode call = conv + SiLU + L2 norms + gates + the
delta rule + the output norm for every (sequence, head).  The other
workloads (varlen prefill, long prefill, verify window + commit) are measured
once more in the same run and reported under "legs".

Timing: W untimed warm-up steps, then exactly K steps timed with CUDA events
on the launching stream, bracketed by a barrier and a device synchronise on
both sides; the max over ranks is reported.  Inputs rotate over several
sets whose total footprint is well above the 129 MB L2, so every step reads
its state from HBM.  Under torchrun each rank runs its own batch (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), float(
            d.get("bf16_tflops_sustained", d.get("bf16_tflops", FALLBACK_BF16_TFLOPS))), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kda_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "power_w_max": max(r[2] for r in rows), "reasons": reasons}


_FLUSH = {}
L2_NOTE = "flushed before each timed call (a read of twice the L2 size)"


def l2_flush():
    """Read a buffer of twice the L2 size and wait for it, outside any timed
    region: whatever a set-up step left in L2 (states just reset, a previous
    call's outputs) is evicted -- dirty lines written back now, not during the
    next timed kernel -- and that kernel reads its inputs from HBM."""
    import torch

    buf = _FLUSH.get("buf")
    if buf is None:
        buf = _FLUSH["buf"] = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    _FLUSH["sink"] = buf.sum()
    torch.cuda.synchronize()


def time_steps(fn, steps, stream, queue_ahead=True, per_step=True):
    """Per-step CUDA-event durations (ms) of fn(i) on `stream`, and the
    elapsed time of the whole sequence.  With queue_ahead the stream first
    sleeps on the GPU so the host can enqueue every step before the GPU
    reaches the first one: the events then time GPU execution, not host
    launch overhead (which the end-to-end figure measures).  Without
    per_step only the first start and the last end are recorded (an event
    between back-to-back launches adds a gap of its own); every step's
    duration is then reported as the elapsed time over the steps."""
    import torch

    n_ev = steps if per_step else 1
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    if queue_ahead:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(2e6) + 200000 * steps)
    for i in range(steps):
        if per_step or i == 0:
            starts[i if per_step else 0].record(stream)
        fn(i)
        if per_step or i == steps - 1:
            ends[i if per_step else 0].record(stream)
    torch.cuda.synchronize()
    total = starts[0].elapsed_time(ends[-1])
    if not per_step:
        return [total / steps] * steps, total
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], total


# ------------------------------------------------------- algorithmic bytes

def decode_bytes_per_unit(d=128, K=4, io=2, out=2, out_gate=True):
    """HBM bytes one (sequence, head) decode row must move: state read and
    write, the q/k/v/gate rows, beta, the output gate, the output, and the
    conv state's K-1 rows read and written."""
    conv = (K - 1) * 3 * d * io
    return 2 * d * d * 4 + 4 * d * io + io + (d * io if out_gate else 0) + d * out + 2 * conv


def prefill_bytes_per_token_head(d=128, io=2, out=4, out_gate=False):
    """HBM bytes per (row, head) of a fully fused prefill: raw q, k, v, gate
    rows and beta in, the output out (states amortised over the sequence)."""
    return 4 * d * io + io + (d * io if out_gate else 0) + d * out


def prefill_state_bytes(N, H, d=128, K=4, io=2):
    return N * H * (2 * d * d * 4 + 2 * (K - 1) * 3 * d * io)


# --------------------------------------------------------------- workloads

class nvtx_range:
    """An NVTX range around a leg of the benchmark (shows in nsys/ncu
    timelines; a no-op without a profiler)."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        import torch

        torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        import torch

        torch.cuda.nvtx.range_pop()
        return False


_WL_CACHE = {}


def cached(wl_fn):
    """The workload wl_fn() builds, drawn once per run (the full-size draws
    take seconds)."""
    if wl_fn not in _WL_CACHE:
        _WL_CACHE[wl_fn] = wl_fn()
    return _WL_CACHE[wl_fn]


def make_sets(wl_fn, n_sets, out_dtype):
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    sets = []
    wl = wl_fn()
    for _ in range(n_sets):
        sets.append(DeviceCase(wl, out_dtype=out_dtype))
    return wl, sets


def bench_decode(kda, steps, warmup, stream):
    from linear_attention_serving_kda_gb300 import workloads as W

    wl = W.decode_case()
    per_set = decode_bytes_per_unit() * wl.N * wl.H
    n_sets = max(3, int(np.ceil(3 * L2_BYTES / per_set)))
    _, sets = make_sets(W.decode_case, n_sets, W.BF16)
    calls = [kda.Prepared("kda_decode", s.params(), wl.N, s.q, s.k, s.v, s.f, s.b, s.g, None,
                          s.conv_state, s.rec_state, s.out, s.dev_status, stream=stream) for s in sets]

    def step(i):
        if calls[i % n_sets]() != 0:
            raise RuntimeError("kda_decode failed")

    for i in range(warmup):
        step(i)
    return wl, sets, step, per_set


def max_over_ranks(x: float, dist) -> float:
    """The largest of every rank's x (the job is as slow as its slowest rank)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank_step: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch each step."""
    return tokens_per_rank_step * world * steps / (total_ms * 1e-3)


def run_timed(step, steps, stream, dist):
    """The timed region: K decode steps (one kernel launch each) between two
    events; a launch's duration is taken as the region over K (gaps between
    launches included)."""
    import torch

    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    durs, total_ms = time_steps(step, steps, stream, per_step=False)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    return max_over_ranks(total_ms, dist), durs, wall


def leg_prefill(kda, wl_fn, reps, stream):
    import torch

    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = cached(wl_fn)
    dc = DeviceCase(wl, out_dtype=W.BF16)
    kda.check(dc.prefill(stream=stream))  # warm-up
    durs = []
    for _ in range(reps):
        dc.reset_states()
        l2_flush()
        durs += time_steps(lambda i: kda.check(dc.prefill(stream=stream)), 1, stream)[0]
    ms = statistics.median(durs)
    bpt = prefill_bytes_per_token_head(out=2, out_gate=wl.has_out_gate)
    alg = wl.T * wl.H * bpt + prefill_state_bytes(wl.N, wl.H)
    # algorithmic tensor work: 5 C d + 6 d^2 FLOPs per (row, head) (chunk C = 64;
    # triangles at half), against the measured dense bf16 tensor peak (burst:
    # the kernel is timed alone).  tf32_frac is a secondary figure: the same
    # FLOPs against the tf32 rate (nominally half of bf16's) that the first
    # two products run at.
    d = wl.dk
    flops = wl.T * wl.H * (5 * 64 * d + 6 * d * d)
    bf16_tflops = load_peaks()[1]
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": wl.name, "tokens": wl.T, "ms": ms, "tokens_per_s": wl.T / (ms * 1e-3),
            "alg_bytes": alg, "achieved_gbs": alg / (ms * 1e-3) / 1e9,
            "alg_flops": flops, "alg_tflops": tf, "bf16_frac": tf / bf16_tflops,
            "bf16_frac_of": f"measured bf16 dense burst peak {bf16_tflops} TFLOP/s",
            "tf32_frac": tf / (bf16_tflops / 2.0), "l2": L2_NOTE}


def leg_prefill_scan(kda, wl_fn, segments, reps, stream):
    """The same prefill through kda_prefill_scan (the affine state scan over
    `segments` pieces per sequence): time per call and tokens/s."""
    import torch

    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = cached(wl_fn)
    dc = DeviceCase(wl, out_dtype=W.BF16)
    p = dc.params()
    need = kda.kda_prefill_scan_workspace_bytes(p, wl.N, wl.T, segments)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(i):
        kda.check(kda.kda_prefill_scan(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, dc.g, None,
                                       dc.conv_state, dc.rec_state, dc.out, ws, need, segments, dc.dev_status,
                                       stream))

    call(0)  # warm-up
    durs = []
    for _ in range(reps):
        dc.reset_states()
        l2_flush()
        durs += time_steps(call, 1, stream)[0]
    ms = statistics.median(durs)
    return {"workload": wl.name, "segments": segments, "tokens": wl.T, "ms": ms,
            "tokens_per_s": wl.T / (ms * 1e-3), "workspace_bytes": need, "l2": L2_NOTE}


def leg_verify(kda, reps, stream):
    import torch

    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = W.verify_case()
    n_sets = 4
    sets = [DeviceCase(wl, out_dtype=W.BF16) for _ in range(n_sets)]
    for s in sets:
        s.alloc_log()
    logs2 = [torch.empty_like(s.log) for s in sets]
    tv, tc, tcv = [], [], []
    for r in range(reps + 1):
        s = sets[r % n_sets]
        s.reset_states()
        l2_flush()  # each timed call reads its states and rows from HBM
        dv = time_steps(lambda i: kda.check(s.verify(stream=stream)), 1, stream)[0]
        l2_flush()
        dcm = time_steps(lambda i: kda.check(s.commit(stream=stream)), 1, stream)[0]
        # the next window in one call: commit this window's accepted rows, verify new rows
        p = s.params()
        lg2 = logs2[r % n_sets]
        l2_flush()
        dcv = time_steps(lambda i: kda.check(kda.kda_commit_verify(
            p, wl.N, wl.W, s.accepted, s.log, s.q, s.k, s.v, s.f, s.b, s.g, s.slots, s.conv_state,
            s.rec_state, lg2, s.out, s.dev_status, stream)), 1, stream)[0]
        if r:
            tv += dv
            tc += dcm
            tcv += dcv
    mv, mc, mcv = statistics.median(tv), statistics.median(tc), statistics.median(tcv)
    acc = int(wl.arrays["accepted"].sum())
    rows = wl.N * wl.W
    # algorithmic HBM bytes per launch (each state, row, log entry moved once)
    io, d, H, Wn, K = 2, wl.dk, wl.H, wl.W, wl.K
    state = d * d * 4
    conv = (K - 1) * 3 * d * io                                  # one head's conv history
    row_in = (4 * d + 1) * io + (d * io if wl.has_out_gate else 0)  # q, k, v, f, beta (, g)
    row_io = row_in + d * 2 + 3 * d * 4 + 3 * d * io             # + bf16 out + log (alpha|k^|u, raw row)
    per_acc = [int(x) for x in wl.arrays["accepted"]]
    v_bytes = wl.N * H * (state + conv + Wn * row_io)
    c_bytes = sum(H * (2 * state + a * 3 * d * 4 + 2 * conv) for a in per_acc if a > 0)
    cv_bytes = v_bytes + sum(H * (state + a * 3 * d * 4 + conv) for a in per_acc if a > 0)
    hbm_gbs = load_peaks()[0]
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    return {"workload": wl.name, "rows": rows, "accepted_rows": acc, "verify_ms": mv, "commit_ms": mc,
            "commit_verify_ms": mcv,
            "rows_verified_per_s": rows / (mv * 1e-3),
            "committed_tokens_per_s": acc / ((mv + mc) * 1e-3),
            "committed_tokens_per_s_fused": acc / (mcv * 1e-3),
            "alg_bytes": {"verify": v_bytes, "commit": c_bytes, "commit_verify": cv_bytes},
            "hbm_frac": {"verify": gbs(v_bytes, mv) / hbm_gbs, "commit": gbs(c_bytes, mc) / hbm_gbs,
                         "commit_verify": gbs(cv_bytes, mcv) / hbm_gbs}, "l2": L2_NOTE}


def e2e_decode(kda, steps, warmup, stream):
    """Same decode step through the public API, host buffers, as a serving
    loop runs it: each step's rows come from pinned host memory (q, k, v,
    gate, beta and output gate packed back to back, one host-to-device copy)
    and its output goes back to pinned host memory, both inside the timed
    region.  The copies run on their own streams, double-buffered, so the
    upload of step i+1 and the download of step i overlap the decode of step
    i; events order each buffer's reuse.  The call is a pre-marshalled
    `kda.Prepared` decode on the device copy of the step's rows.  The timed
    region runs from before the first upload to the end of the last
    download, host launch overhead included (no queue-ahead)."""
    import torch

    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = W.decode_case()
    dc = DeviceCase(wl, out_dtype=W.BF16)
    names = ("q", "k", "v", "f", "b", "g")
    srcs = {nm: wl.to_torch(nm) for nm in names}
    offs, off = {}, 0
    for nm in names:
        offs[nm] = off
        off += (srcs[nm].numel() * srcs[nm].element_size() + 255) // 256 * 256

    def view(buf, nm):
        t = srcs[nm]
        n = t.numel() * t.element_size()
        return buf[offs[nm]:offs[nm] + n].view(t.dtype).view(t.shape)

    NB = 2
    host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    for nm in names:
        view(host_in, nm).copy_(srcs[nm])
    dev_in = [torch.empty(off, dtype=torch.uint8, device="cuda") for _ in range(NB)]
    dev_out = [torch.empty_like(dc.out) for _ in range(NB)]
    host_out = [torch.empty(dc.out.shape, dtype=dc.out.dtype).pin_memory() for _ in range(NB)]
    h2d = sum(srcs[nm].numel() * srcs[nm].element_size() for nm in names)
    d2h = host_out[0].numel() * host_out[0].element_size()
    calls = []
    for j in range(NB):
        dv = {nm: view(dev_in[j], nm) for nm in names}
        calls.append(kda.Prepared("kda_decode", dc.params(), wl.N, dv["q"], dv["k"], dv["v"], dv["f"], dv["b"],
                                  dv["g"], None, dc.conv_state, dc.rec_state, dev_out[j], dc.dev_status,
                                  stream=stream))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    uploaded = [ev() for _ in range(NB)]   # rows of buffer j on the device
    computed = [ev() for _ in range(NB)]   # decode on buffer j done (rows free, output ready)
    fetched = [ev() for _ in range(NB)]    # output of buffer j copied back (output free)

    def step(i):
        j = i % NB
        with torch.cuda.stream(up):
            if i >= NB:
                up.wait_event(computed[j])
            dev_in[j].copy_(host_in, non_blocking=True)
            uploaded[j].record(up)
        stream.wait_event(uploaded[j])
        if i >= NB:
            stream.wait_event(fetched[j])
        kda.check(calls[j]())
        computed[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[j])
            host_out[j].copy_(dev_out[j], non_blocking=True)
            fetched[j].record(down)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for i in range(steps):
        step(i)
    stream.wait_stream(down)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": wl.N / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipeline": "upload of step i+1 and download of step i overlap the decode of step i"}


def _pack_rows(dc, names):
    """Pack a DeviceCase's row tensors back to back (256-byte aligned pieces)
    into one pinned host buffer and one device buffer, and rebind the case's
    tensors to views of the device buffer, so that one host-to-device copy
    brings in every input row of a call.  Returns (host, device, h2d bytes)."""
    import torch

    offs, off = {}, 0
    for nm in names:
        t = getattr(dc, nm)
        offs[nm] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev = torch.empty(off, dtype=torch.uint8, device="cuda")
    n_bytes = 0
    for nm in names:
        t = getattr(dc, nm)
        n = t.numel() * t.element_size()
        host[offs[nm]:offs[nm] + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        setattr(dc, nm, dev[offs[nm]:offs[nm] + n].view(t.dtype).view(t.shape))
        n_bytes += n
    return host, dev, n_bytes


def e2e_leg(kda, dc, names, call, out_view, reps, stream):
    """A leg's call end to end through the public API with host buffers: each
    rep copies the call's input rows from pinned host memory (one packed
    copy), runs `call()` on them and copies `out_view()` back to pinned host
    memory, all on `stream` and inside the CUDA-event region.  States stay
    resident (reset between reps, outside the region).  Median over reps."""
    import torch

    host, dev, h2d = _pack_rows(dc, names)
    out_host = torch.empty(out_view().shape, dtype=out_view().dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    durs = []
    for r in range(reps + 1):
        dc.reset_states()
        l2_flush()  # the states come from HBM, as after other work in a serving loop
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            dev.copy_(host, non_blocking=True)
            kda.check(call())
            out_host.copy_(out_view(), non_blocking=True)
            t1.record(stream)
        torch.cuda.synchronize()
        if r:  # the first rep warms up
            durs.append(t0.elapsed_time(t1))
    return statistics.median(durs), h2d, d2h


def e2e_prefill(kda, wl_fn, reps, stream):
    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = cached(wl_fn)
    dc = DeviceCase(wl, out_dtype=W.BF16)
    names = ["q", "k", "v", "f", "b"] + (["g"] if wl.has_out_gate else [])
    ms, h2d, d2h = e2e_leg(kda, dc, names, lambda: dc.prefill(stream=stream), lambda: dc.out[:wl.T], reps, stream)
    return {"value": wl.T / (ms * 1e-3), "unit": "tokens/s", "ms": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "path": "kda_prefill_varlen: rows host->device, prefill, outputs device->host"}


def e2e_prefill_pipelined(kda, wl_fn, pieces, reps, stream):
    """The same prefill end to end as a serving loop would overlap it: the
    batch is cut into `pieces` -- whole-sequence groups (balanced by rows) for
    a varlen batch, consecutive 64-row-aligned cuts of the prompt (state
    carried from one cut to the next) for a single sequence -- each piece's
    rows are uploaded from pinned host memory on a copy stream, each piece is
    prefilled as soon as its rows are on the device (groups on streams of
    their own, cuts in order on one stream), and each piece's outputs are
    copied back as soon as it is done.  The CUDA-event region spans the first
    upload to the last download; states stay resident and are reset outside it.
    A prompt cut at multiples of 64 rows gives the uncut call's bits (bounded
    gates), so the cuts change only the schedule."""
    import torch

    from linear_attention_serving_kda_gb300 import shard
    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = cached(wl_fn)
    names = ["q", "k", "v", "f", "b"] + (["g"] if wl.has_out_gate else [])
    if wl.N > 1:
        groups = [g for g in shard.partition_sequences(wl.cu_seqlens, pieces) if g]
        subs = [shard.shard_workload(wl, g) for g in groups]
        chained = False
    else:
        subs = [shard.cut_prompt(wl, a, b) for a, b in shard.prompt_cuts(wl.T, pieces)]
        chained = True
    cases = [DeviceCase(sw, out_dtype=W.BF16) for sw in subs]
    if chained:  # the cuts carry one sequence's states
        for dc in cases[1:]:
            dc.conv_state, dc.rec_state = cases[0].conv_state, cases[0].rec_state
    packs = [_pack_rows(dc, names) for dc in cases]
    outs = [torch.empty(dc.out[:dc.wl.T].shape, dtype=dc.out.dtype).pin_memory() for dc in cases]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    comp = [stream] if chained else [torch.cuda.Stream() for _ in cases]
    for dc in cases:  # workspaces allocated outside the timed region
        dc.prefill(stream=stream)
    torch.cuda.synchronize()
    durs = []
    for r in range(reps + 1):
        for dc in cases[:1] if chained else cases:  # the cuts share the first case's states
            dc.reset_states()
        l2_flush()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(up)
        for i, (dc, (host, dev, _)) in enumerate(zip(cases, packs)):
            ev_up, ev_done = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(up):
                dev.copy_(host, non_blocking=True)
                ev_up.record(up)
            cs = comp[0] if chained else comp[i]
            cs.wait_event(ev_up)
            kda.check(dc.prefill(stream=cs))
            ev_done.record(cs)
            with torch.cuda.stream(down):
                down.wait_event(ev_done)
                outs[i].copy_(dc.out[:dc.wl.T], non_blocking=True)
        t1.record(down)
        torch.cuda.synchronize()
        if r:
            durs.append(t0.elapsed_time(t1))
    ms = statistics.median(durs)
    h2d = sum(p[2] for p in packs)
    d2h = sum(o.numel() * o.element_size() for o in outs)
    return {"value": wl.T / (ms * 1e-3), "unit": "tokens/s", "ms": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "pieces": len(cases),
            "path": ("kda_prefill_varlen per group of whole sequences" if not chained else
                     "kda_prefill_varlen per 64-row-aligned cut, state carried") +
                    ": each piece's upload, call and download overlapped with the others'"}


def e2e_verify(kda, reps, stream):
    from linear_attention_serving_kda_gb300 import workloads as W
    from linear_attention_serving_kda_gb300.runtime import DeviceCase

    wl = W.verify_case()
    dc = DeviceCase(wl, out_dtype=W.BF16)
    dc.alloc_log()
    names = ["q", "k", "v", "f", "b", "accepted"] + (["g"] if wl.has_out_gate else [])

    def call():
        rc = dc.verify(stream=stream)
        return rc if rc != 0 else dc.commit(stream=stream)

    ms, h2d, d2h = e2e_leg(kda, dc, names, call, lambda: dc.out[:wl.N * wl.W], reps, stream)
    acc = int(wl.arrays["accepted"].sum())
    return {"value": wl.N * wl.W / (ms * 1e-3), "unit": "rows verified/s", "ms": ms,
            "committed_tokens_per_s": acc / (ms * 1e-3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "window rows and accepted counts host->device, kda_verify_window + kda_commit, "
                    "window outputs device->host"}


# --------------------------------------------------------- CPU oracle legs

def oracle_decode_rate(seconds=10.0):
    """The oracle (threads over (sequence, head) units, as it stands) on the
    decode step, repeated with carried states for about `seconds`."""
    import oracle
    from linear_attention_serving_kda_gb300 import workloads as W

    oracle.build()
    wl = W.decode_case()
    cores = os.cpu_count() or 1
    steps = 0
    t0 = time.perf_counter()
    arrays = dict(wl.arrays)
    while True:
        res = oracle.forward(wl, threads=cores, arrays=arrays)
        arrays["rec_state"], arrays["conv_state"] = res["rec_state"], res["conv_state"]
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return wl.N * steps / el, cores, steps, el


def oracle_decode_rate_1thread(seconds=1.0):
    """The oracle on one thread: all heads of one sequence's decode row,
    repeated for about `seconds`; tokens/s = rows (all heads) per second."""
    import oracle
    from linear_attention_serving_kda_gb300 import shard, workloads as W

    oracle.build()
    one = shard.shard_workload(W.decode_case(), [0])  # sequence 0: its row, states and the parameters
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.forward(one, threads=1)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return n / el, n, el


def oracle_units_rate(wl, units, rows, threads):
    """Row-heads per second of the oracle (as it stands) over the given
    (sequence, head) units of a workload, each cut to its first `rows` rows
    (pure data movement), run on `threads` threads."""
    import oracle
    from linear_attention_serving_kda_gb300 import shard, workloads as W

    oracle.build()
    subs = []
    for s, h in units:
        sub = W.head_slice(wl, s, h)
        if rows is not None and sub.T > rows:
            sub = shard.cut_prompt(sub, 0, rows)
        subs.append(sub)
    work = sum(sb.T for sb in subs)
    from concurrent.futures import ThreadPoolExecutor

    t0 = time.perf_counter()
    if threads <= 1:
        for sb in subs:
            oracle.forward(sb, threads=1)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda sb: oracle.forward(sb, threads=1), subs))
    el = time.perf_counter() - t0
    return work / el, work, el


def oracle_leg_baseline(wl, rows, per_thread_units=1):
    """The oracle on a bounded sample of a leg's own workload: one
    (sequence, head) unit per host core (cut to `rows` rows) on all cores,
    and one unit on one thread.  tokens/s = row-heads/s / H."""
    cores = os.cpu_count() or 1
    n = cores * per_thread_units
    units = [(i % wl.N, (i // wl.N) % wl.H) for i in range(n)]
    rate_mt, work_mt, el_mt = oracle_units_rate(wl, units, rows, cores)
    rate_1, work_1, el_1 = oracle_units_rate(wl, units[:1], 2048 if rows is None else min(rows, 2048), 1)
    return {"value": rate_mt / wl.H, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "value_1thread": rate_1 / wl.H,
            "sample": f"{len(units)} (sequence, head) units of {wl.name}, "
                      f"{'whole' if rows is None else f'each its first {rows} rows'} "
                      f"({work_mt} row-heads in {el_mt:.1f} s on {cores} threads; 1 thread: {work_1} row-heads "
                      f"in {el_1:.1f} s); tokens/s = row-heads/s / {wl.H} heads"}


def oracle_verify_baseline(seconds_hint=None):
    """The oracle on the verify workload: the window rows of every (sequence,
    head) unit (the verify step) on all cores, and on one thread over the
    first unit's window repeated."""
    import oracle
    from linear_attention_serving_kda_gb300 import workloads as W

    oracle.build()
    wl = W.verify_case()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.forward(wl, threads=cores)
    el = time.perf_counter() - t0
    rows = wl.N * wl.W
    sub = W.head_slice(wl, 0, 0)
    t1 = time.perf_counter()
    reps = 64
    for _ in range(reps):
        oracle.forward(sub, threads=1)
    el1 = time.perf_counter() - t1
    return {"value": rows / el, "unit": "rows verified/s", "cores": cores, "kind": "oracle",
            "value_1thread": reps * wl.W / el1 / wl.H,
            "sample": f"the whole verify window ({wl.N} x {wl.W} rows x {wl.H} heads) in {el:.2f} s on {cores} "
                      f"threads; 1 thread: one (sequence, head) window x {reps} in {el1:.2f} s, scaled by 1/{wl.H}"}


def measured_traffic():
    """DRAM bytes per decode launch from the committed ncu record, or None
    when the kernel source has changed since the counters were taken."""
    import hashlib

    tpath = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(tpath) as fh:
            rec = json.load(fh)
        h = hashlib.sha256()
        for src in rec["sources"]:  # the kernel's source files, in this order
            with open(os.path.join(ROOT, src), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


# --------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-legs", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "verify", "prefill_varlen", "prefill_long", "prefill_small",
                             "prefill_varlen_softplus", "prefill_long_scan", "prefill_scan_small",
                             "e2e_prefill_varlen", "e2e_prefill_long"])
    ap.add_argument("--segments", type=int, default=4,
                    help="segments of the prompt for prefill_long_scan; pieces for the e2e_prefill_* workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: run this same command under torchrun
        import socket

        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and rank == 0:
        print(f"bench.py: --gpus {args.gpus} but {world} ranks were launched; measuring {world}", file=sys.stderr)

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, world)
        return

    import torch

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist

    import linear_attention_serving_kda_gb300 as kda
    from linear_attention_serving_kda_gb300 import build as kbuild

    if rank == 0 or world == 1:
        kbuild.build()
    if dist is not None:
        dist.barrier()
    kda.load()
    stream = torch.cuda.current_stream()  # every launch and every event goes on this stream
    hbm_gbs, _, _, peak_src = load_peaks()
    sampler = ClockSampler(local_rank).start() if rank == 0 else None

    if args.workload != "decode":
        res = run_single_leg(kda, args, stream)
        if sampler:
            res["clocks"] = sampler.stop()
        if rank == 0:
            print(json.dumps(res))
        return

    with nvtx_range("decode warm-up"):
        wl, sets, step, per_set = bench_decode(kda, args.steps, args.warmup, stream)
    with nvtx_range("decode timed"):
        total_ms, durs, _ = run_timed(step, args.steps, stream, dist)
    ms = total_ms / args.steps
    value = weak_scaling_value(wl.N, world, args.steps, total_ms)
    kernel_ms = statistics.mean(durs)
    achieved = per_set / (kernel_ms * 1e-3) / 1e9

    legs = {}
    if not args.no_legs:
        from linear_attention_serving_kda_gb300 import workloads as W

        with nvtx_range("leg prefill_varlen"):
            legs["prefill_varlen"] = leg_prefill(kda, W.varlen_prefill_case, 3, stream)
        with nvtx_range("leg prefill_long"):
            legs["prefill_long"] = leg_prefill(kda, W.long_prefill_case, 3, stream)
        with nvtx_range("leg verify_commit"):
            legs["verify_commit"] = leg_verify(kda, 10, stream)
        with nvtx_range("leg prefill_long_scan"):
            legs["prefill_long_scan"] = leg_prefill_scan(kda, W.long_prefill_case, 4, 3, stream)
        for k in ("prefill_varlen", "prefill_long"):
            legs[k]["hbm_frac"] = legs[k]["achieved_gbs"] / hbm_gbs
        with nvtx_range("legs end to end"):
            legs["prefill_varlen"]["e2e"] = e2e_prefill(kda, W.varlen_prefill_case, 5, stream)
            legs["prefill_long"]["e2e"] = e2e_prefill(kda, W.long_prefill_case, 5, stream)
            legs["verify_commit"]["e2e"] = e2e_verify(kda, 10, stream)
            legs["prefill_varlen"]["e2e_pipelined"] = e2e_prefill_pipelined(kda, W.varlen_prefill_case, 8, 5,
                                                                            stream)
            legs["prefill_long"]["e2e_pipelined"] = e2e_prefill_pipelined(kda, W.long_prefill_case, 16, 5, stream)
    with nvtx_range("decode end to end"):
        e2e = e2e_decode(kda, args.steps, args.warmup, stream)
    e2e["value"] *= world
    clocks = sampler.stop() if sampler else None

    cpu = None
    if rank == 0 and world == 1:
        rate, cores, n, el = oracle_decode_rate(args.cpu_seconds)
        rate1, n1, el1 = oracle_decode_rate_1thread(max(0.1, args.cpu_seconds / 10))
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "value_1thread": rate1,
               "sample": f"full decode step (64 seq x 32 heads) repeated {n}x with carried state, {el:.1f} s; "
                         f"1 thread: one sequence's row through all 32 heads x {n1} in {el1:.2f} s"}

    if rank == 0 and world == 1 and legs and args.cpu_seconds > 0:
        from linear_attention_serving_kda_gb300 import workloads as W

        legs["prefill_varlen"]["cpu_baseline"] = oracle_leg_baseline(cached(W.varlen_prefill_case), None, 2)
        legs["prefill_long"]["cpu_baseline"] = oracle_leg_baseline(cached(W.long_prefill_case), 8192, 2)
        legs["verify_commit"]["cpu_baseline"] = oracle_verify_baseline()

    traffic = measured_traffic()

    line = {
        "metric": "KDA tokens/s (decode step; prefill and verify legs alongside)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.N, "heads": wl.H, "head_dim": wl.dk,
                   "conv_kernel": wl.K, "io": "bf16", "state": "fp32", "gate": "softplus",
                   "epilogue": "sigmoid-gated RMSNorm", "parallelism": f"replica x{world}",
                   "l2": f"inputs rotate over {len(sets)} sets, {len(sets) * per_set / 1e6:.0f} MB > L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": traffic, "kernel": "kda_decode_stream_kernel<bf16>",
                     "alg_bytes_per_launch": per_set, "peak_source": peak_src, "launch_ms": kernel_ms,
                     "launch_ms_from": "CUDA events around the K timed launches, divided by K"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "legs": legs,
    }
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_single_leg(kda, args, stream):
    from linear_attention_serving_kda_gb300 import workloads as W

    if args.workload == "verify":
        return leg_verify(kda, args.steps, stream)
    if args.workload == "prefill_long_scan":
        return leg_prefill_scan(kda, W.long_prefill_case, args.segments, args.steps, stream)
    if args.workload in ("e2e_prefill_varlen", "e2e_prefill_long"):
        fn = W.varlen_prefill_case if args.workload == "e2e_prefill_varlen" else W.long_prefill_case
        return {"serial": e2e_prefill(kda, fn, args.steps, stream),
                "pipelined": e2e_prefill_pipelined(kda, fn, args.segments, args.steps, stream)}
    if args.workload == "prefill_scan_small":
        # a profiling-sized prompt for the scan path: 1 sequence x 8192 rows, the long prompt's dtypes and gate
        fn = lambda: W.long_prefill_case(8192)  # noqa: E731
        return leg_prefill_scan(kda, fn, args.segments, args.steps, stream)
    if args.workload == "prefill_small":
        # a profiling-sized prefill: 2 sequences x 2048 rows, 32 heads, same dtypes and gate
        fn = lambda: W.make_workload("prefill_small_n2x2048_h32_d128_bf16", 5, [2048, 2048], H=32, d=128,  # noqa: E731
                                     K=4, io_dtype=W.BF16, gate_mode=W.SAFE, lower_bound=-5.0,
                                     init_state="random")
        return leg_prefill(kda, fn, args.steps, stream)
    if args.workload == "prefill_varlen_softplus":
        # the varlen case's lengths and rows with the softplus gate: the chunk
        # kernel's data-dependent chunks
        fn = lambda: W.make_workload("prefill_varlen_softplus_n8_h32_d128_bf16", 2, None, H=32, d=128,  # noqa: E731
                                     K=4, io_dtype=W.BF16, gate_mode=W.SOFTPLUS, lower_bound=-5.0,
                                     init_state="random", draw_lens=(8, 512, 8192))
        return leg_prefill(kda, fn, args.steps, stream)
    fn = W.varlen_prefill_case if args.workload == "prefill_varlen" else W.long_prefill_case
    return leg_prefill(kda, fn, args.steps, stream)


def run_reference(args, world):
    """The fp64 oracle on the host cores, same workload, metric and unit."""
    from linear_attention_serving_kda_gb300 import workloads as W
    import oracle

    oracle.build()
    wl = W.decode_case()
    cores = os.cpu_count() or 1
    arrays = dict(wl.arrays)
    for _ in range(args.warmup):
        res = oracle.forward(wl, threads=cores, arrays=arrays)
        arrays["rec_state"], arrays["conv_state"] = res["rec_state"], res["conv_state"]
    t0 = time.perf_counter()
    for _ in range(args.steps):
        res = oracle.forward(wl, threads=cores, arrays=arrays)
        arrays["rec_state"], arrays["conv_state"] = res["rec_state"], res["conv_state"]
    el = time.perf_counter() - t0
    value = wl.N * args.steps / el
    line = {
        "impl": "reference",
        "metric": "KDA tokens/s (decode step; prefill and verify legs alongside)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.N, "heads": wl.H, "head_dim": wl.dk,
                   "conv_kernel": wl.K, "io": "bf16", "state": "fp64 (oracle)", "gate": "softplus"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"full decode step x {args.steps} with carried state"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
