"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import linear_attention_serving_kda_gb300 as kda
from linear_attention_serving_kda_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")
FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced here


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"kda_prefill_varlen", "kda_decode", "kda_verify_window", "kda_commit", "kda_commit_verify"} <= set(names)
    raw = ctypes.CDLL(kbuild.LIB)
    for n in names:
        assert hasattr(raw, n), n
    assert lib.kda_abi_version() == 100


def _params(**kw):
    base = dict(num_heads=4, head_dim=128, conv_kernel=4, gate_mode=kda.KDA_GATE_SAFE,
                A_log=FAKE, dt_bias=FAKE, conv_weight=FAKE, gate_lower_bound=-5.0, num_slots=4)
    base.update(kw)
    return kda.Params(**base)


def _decode(p, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, gate=FAKE, beta=FAKE, out_gate=None, slots=None,
                conv_state=FAKE, rec_state=FAKE, out=FAKE)
    args.update(over)
    return kda.kda_decode(p, 2, args["q"], args["k"], args["v"], args["gate"], args["beta"],
                          args["out_gate"], args["slots"], args["conv_state"], args["rec_state"],
                          args["out"], None, 0)


@pytest.mark.parametrize("kw,rc", [
    (dict(head_dim=96), kda.KDA_ERR_UNSUPPORTED_GEOMETRY),
    (dict(head_dim=256), kda.KDA_ERR_UNSUPPORTED_GEOMETRY),
    (dict(head_dim_v=64), kda.KDA_ERR_UNSUPPORTED_GEOMETRY),
    (dict(conv_kernel=5), kda.KDA_ERR_UNSUPPORTED_GEOMETRY),
    (dict(conv_kernel=1), kda.KDA_ERR_UNSUPPORTED_GEOMETRY),
    (dict(gate_lower_bound=0.0), kda.KDA_ERR_INVALID_BOUND),
    (dict(gate_lower_bound=float("nan")), kda.KDA_ERR_INVALID_BOUND),
    (dict(gate_lower_bound=float("-inf")), kda.KDA_ERR_INVALID_BOUND),
    (dict(gate_mode=7), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(num_heads=0), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(num_slots=0), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(io_dtype=5), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(l2_eps=-1.0), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("inf")), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(A_log=None), kda.KDA_ERR_INVALID_ARGUMENT),
    (dict(dt_bias=FAKE + 4), kda.KDA_ERR_INVALID_ARGUMENT),
])
def test_params_rejected_before_launch(lib, kw, rc):
    assert _decode(_params(**kw)) == rc


def test_bound_checked_only_in_safe_mode(lib):
    # a positive bound is irrelevant to the softplus gate: the parameters pass
    # validation and the call fails only at the pointer check that follows
    # (a null q row pointer) -- before any launch, so the placeholder
    # addresses are never handed to a kernel, with or without a GPU
    p = _params(gate_mode=kda.KDA_GATE_SOFTPLUS, gate_lower_bound=3.0)
    assert _decode(p, q=None) == kda.KDA_ERR_INVALID_ARGUMENT
    assert _decode(_params(gate_lower_bound=3.0), q=None) == kda.KDA_ERR_INVALID_BOUND


def test_pointer_checks(lib):
    p = _params()
    assert _decode(p, q=None) == kda.KDA_ERR_INVALID_ARGUMENT
    assert _decode(p, out=FAKE + 2) == kda.KDA_ERR_INVALID_ARGUMENT
    assert _decode(p, out_gate=FAKE + 8) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_decode(p, -1, *([FAKE] * 5), None, None, FAKE, FAKE, FAKE, None, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_decode(p, 0, *([None] * 10), None, 0) == kda.KDA_OK  # empty batch: no-op
    # prefill: zero sequences is a no-op; negative sizes are rejected
    assert kda.kda_prefill_varlen(p, None, 0, 0, *([None] * 10), None, 0, None, 0) == kda.KDA_OK
    assert kda.kda_prefill_varlen(p, FAKE, -1, 0, *([None] * 10), None, 0, None, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_verify_window(p, 2, 4, *([FAKE] * 5), None, None, FAKE, FAKE, None, FAKE, None, 0) \
        == kda.KDA_ERR_INVALID_ARGUMENT  # missing log
    assert kda.kda_commit(p, 2, 4, None, None, FAKE, FAKE, FAKE, None, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    # commit + verify: missing accepted counts, missing previous log, misaligned new log
    cv = dict(accepted=FAKE, log_prev=FAKE, q=FAKE, k=FAKE, v=FAKE, gate=FAKE, beta=FAKE, out_gate=None,
              slots=None, conv_state=FAKE, rec_state=FAKE, log=FAKE, out=FAKE)
    for over in (dict(accepted=None), dict(log_prev=None), dict(log=FAKE + 4), dict(out_gate=FAKE + 8)):
        args = {**cv, **over}
        assert kda.kda_commit_verify(p, 2, 4, *args.values(), None, 0) == kda.KDA_ERR_INVALID_ARGUMENT, over
    assert kda.kda_commit_verify(p, 0, 4, *([None] * 13), None, 0) == kda.KDA_OK  # empty batch: no-op
    assert kda.kda_commit_verify(p, -1, 4, *cv.values(), None, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    # activation hook: unknown function, negative size, null or misaligned arrays; empty is a no-op
    assert kda.kda_debug_activations(4, FAKE, FAKE, 8, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_debug_activations(kda.KDA_ACT_EXP, FAKE, FAKE, -1, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_debug_activations(kda.KDA_ACT_SILU, None, FAKE, 8, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_debug_activations(kda.KDA_ACT_SILU, FAKE, FAKE + 4, 8, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_debug_activations(kda.KDA_ACT_RCP, None, None, 0, 0) == kda.KDA_OK


def test_sizes(lib):
    p = _params(io_dtype=kda.KDA_DTYPE_BF16)
    n = kda.kda_verify_log_bytes(p, 32, 8)
    floats = 32 * 8 * 4 * 3 * 128 * 4
    raw = 32 * 8 * 4 * 3 * 128 * 2
    assert n >= floats + raw and n % 256 == 0
    assert kda.kda_verify_log_bytes(_params(head_dim=96), 32, 8) == 0
    assert kda.kda_prefill_workspace_bytes(p, 8, 1000) % 256 == 0


def test_split_workspace_size(lib):
    """Few long chains (N * H <= 64, T >= 1024 rows) take the split path:
    the schedule, then one release flag per ring slot plus one consumed
    counter per chain, then 8 slots of 147968 bytes per chain (each slot: the
    chain's operand tiles of a chunk as bf16 high and low parts, then U'^T and
    e^{G_C} in fp32), and last the chains' raw outputs for the epilogue
    (fp32 [T][H][128], 1 KiB aligned)."""
    p = _params(io_dtype=kda.KDA_DTYPE_BF16)  # H = 4
    N, nc = 2, 8
    sched = 1024                      # 3 int32 rounded to 256, then to 1 KiB
    flags = 1024                      # nc * 9 int32 = 288 bytes, rounded to 1 KiB
    # -W and Q o e^G (64 x 128), P (64 x 64), (K o e^{G_C - G})^T (128 x 64), hi and lo,
    # 2 bytes each; U'^T (128 x 64 fp32); e^{G_C} (128 fp32)
    slot = 2 * 2 * (64 * 128 + 64 * 128 + 64 * 64 + 128 * 64) + 128 * 64 * 4 + 128 * 4
    assert slot == 147968
    raw = lambda T: -(-(T * 4 * 128 * 4) // 1024) * 1024  # noqa: E731
    assert kda.kda_prefill_workspace_bytes(p, N, 1024) == sched + flags + nc * 8 * slot + raw(1024)
    assert kda.kda_prefill_workspace_bytes(p, N, 1023) == 256          # short: fused path
    assert kda.kda_prefill_workspace_bytes(p, 17, 4096) == 256 * 1     # 68 chains: fused path
    assert kda.kda_prefill_workspace_bytes(_params(io_dtype=kda.KDA_DTYPE_F32, gate_mode=kda.KDA_GATE_SOFTPLUS),
                                           N, 4096) == 0  # fp32 rows: the row path
    # softplus (and safe gates below -5) chunk where the decays require: fused path only
    # softplus (and safe gates below -5): the split path plus each chain's chunk
    # list (a count, up to T chunk starts, the end, the first cut chunk: T + 3
    # int32), 1 KiB aligned
    bnd = -(-(nc * (4096 + 3) * 4) // 1024) * 1024
    for q in (_params(io_dtype=kda.KDA_DTYPE_BF16, gate_mode=kda.KDA_GATE_SOFTPLUS),
              _params(io_dtype=kda.KDA_DTYPE_BF16, gate_lower_bound=-8.0)):
        assert kda.kda_prefill_workspace_bytes(q, N, 4096) == sched + flags + nc * 8 * slot + bnd + raw(4096)
        assert kda.kda_prefill_workspace_bytes(q, N, 1000) == 256   # short: fused path, no list


def test_status_strings(lib):
    for rc in range(7):
        assert kda.status_string(rc).startswith("KDA_")
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"


def test_guard_regions_catch_writes_past_either_end():
    """The guard regions the GPU tests put around every library-written
    buffer: untouched after in-bounds writes, changed by a write one byte
    before the buffer or one element past its end (checked here on host
    memory; the GPU tests use the same class on device memory)."""
    import torch

    from linear_attention_serving_kda_gb300.runtime import GUARD_BYTES, Guarded

    g = Guarded((3, 5), torch.float32, "cpu")
    g.tensor.fill_(1.0)
    assert g.intact()
    g.raw[GUARD_BYTES - 1] = 0
    assert not g.intact()
    g = Guarded((7,), torch.bfloat16, "cpu")
    g.tensor.fill_(2.0)
    assert g.intact()
    g.raw[GUARD_BYTES + 14] = 0  # the first byte after the 7 bf16 values
    assert not g.intact()


def test_no_unsynchronised_per_device_statics():
    """Per-device host set-up (kernel attributes, capability checks, SM
    counts, the built-in scratch address) is safe to reach from several host
    threads at once: it goes through the PerDeviceOnce helper, atomics or a
    mutex, never a plain static array."""
    import glob
    import re

    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "linear_attention_serving_kda_gb300", "csrc")
    plain = re.compile(r"^\s*static\s+(bool|int|signed char|char|void\*)\s+\w+\[")
    for path in glob.glob(os.path.join(csrc, "*.c*")) + glob.glob(os.path.join(csrc, "*.h")):
        with open(path) as fh:
            for i, line in enumerate(fh, 1):
                assert not plain.match(line), f"{os.path.basename(path)}:{i}: plain per-device static: {line.strip()}"


def test_size_queries_from_many_threads(lib):
    """Size queries and status names called from several host threads at once
    give the answers of one thread."""
    from concurrent.futures import ThreadPoolExecutor

    p = _params()

    def q(_):
        return (kda.kda_prefill_workspace_bytes(p, 8, 32768), kda.kda_prefill_workspace_bytes(p, 1, 32768),
                kda.kda_verify_log_bytes(p, 32, 8), lib.kda_status_string(3))

    want = q(None)
    assert want[0] > 0 and want[1] > 0
    with ThreadPoolExecutor(max_workers=16) as ex:
        got = list(ex.map(q, range(256)))
    assert all(g == want for g in got)


def test_plain_c_consumer(lib, tmp_path):
    """include/kda.h compiles as C11 and a C program linked against the
    library calls its host-side entry points (no GPU needed)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cuda_inc = None
    for cand in ("/usr/local/cuda/include", os.path.join(os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/x/x")), "include")):
        if os.path.exists(os.path.join(cand, "cuda_runtime_api.h")):
            cuda_inc = cand
            break
    if cuda_inc is None:
        pytest.skip("CUDA headers not found")
    src = os.path.join(ROOT, "tests", "c_consumer", "kda_c_consumer.c")
    exe = str(tmp_path / "kda_c_consumer")
    libdir = os.path.dirname(kbuild.LIB)
    subprocess.check_call([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                           src, "-o", exe, "-L", libdir, "-lkda", f"-Wl,-rpath,{libdir}"])
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok") >= 10
