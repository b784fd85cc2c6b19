"""The allocation-free prefill entry point, through the C ABI.

kda_prefill_varlen_static_ws serves callers that cannot allocate device
memory: it keeps the chunk kernel's scratch in a fixed array inside the
library instead of taking a caller workspace.  Its results must be those of
kda_prefill_varlen, call after call, with the shared array reused.  This file
is collected last, so a run that stops at the first failure has run every
other test before it.
"""
import pytest
import torch

from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase

pytestmark = pytest.mark.gpu


def _static_call(kda, dc):
    wl = dc.wl
    return kda.kda_prefill_varlen_static_ws(dc.params(), dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b,
                                            dc.g, dc.slots, dc.conv_state, dc.rec_state, dc.out, dc.dev_status)


@pytest.mark.parametrize("lens,og", [([100, 37, 200], True), ([64, 1, 130, 65, 7], False)])
def test_static_workspace_matches_caller_workspace(cuda_lib, lens, og):
    wl = W.make_workload("noalloc", 500 + sum(lens), lens, H=2, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=og, init_state="random")
    # another batch (more sequences, the longest last) that rewrites the shared array's
    # schedule between the two compared calls
    other = W.make_workload("noalloc_other", 77, [3, 9, 40, 65, 129, 200, 300][:len(lens) + 2], H=2, d=128, K=4,
                            io_dtype=W.BF16, gate_mode=W.SAFE, lower_bound=-5.0, init_state="random")
    ref = DeviceCase(wl)
    assert cuda_lib.kda_prefill_workspace_bytes(ref.params(), wl.N, wl.T) > 0  # the chunk path uses scratch
    cuda_lib.check(ref.prefill())
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share the built-in array
        dc = DeviceCase(wl)
        cuda_lib.check(_static_call(cuda_lib, dc))
        torch.cuda.synchronize()
        assert int(dc.dev_status.item()) == 0
        # the same kernel on the same inputs: the same bits
        assert torch.equal(dc.out[:wl.T], ref.out[:wl.T]), f"out, call {call}"
        assert torch.equal(dc.rec_state, ref.rec_state), f"rec_state, call {call}"
        assert torch.equal(dc.conv_state, ref.conv_state)
        oc = DeviceCase(other)
        cuda_lib.check(_static_call(cuda_lib, oc))
        torch.cuda.synchronize()
        assert int(oc.dev_status.item()) == 0


def test_static_workspace_rejects_oversized_batches(cuda_lib):
    cap = cuda_lib.kda_prefill_static_workspace_capacity()
    assert cap == 256 * 1024
    n_max = cap // 4 - 1
    wl = W.make_workload("noalloc_big", 7, [1], H=1, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, init_state="zero")
    dc = DeviceCase(wl)
    p = dc.params()
    assert cuda_lib.kda_prefill_workspace_bytes(p, n_max + 1, 1) > cap
    rc = cuda_lib.kda_prefill_varlen_static_ws(p, dc.cu_seqlens, n_max + 1, 1, dc.q, dc.k, dc.v, dc.f, dc.b,
                                               None, None, dc.conv_state, dc.rec_state, dc.out, dc.dev_status)
    assert rc == cuda_lib.KDA_ERR_WORKSPACE
