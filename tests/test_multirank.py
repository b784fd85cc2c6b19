"""Multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own batch (weak scaling); the only collective is the
max-over-ranks of the timed region, and the whole-job value counts every
rank's tokens against that slowest time.  A varlen batch splits into
per-rank shards of whole sequences whose results, gathered, are those of one
unsharded run."""
import os
import socket

import numpy as np

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist)   # rank 1 is the slow one
    value = bench.weak_scaling_value(64, world, 100, slowest)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == pytest.approx(15.0)
        assert value == pytest.approx(64 * 2 * 100 / 15e-3)


def test_single_rank_needs_no_collective():
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.weak_scaling_value(64, 1, 10, 2.0) == pytest.approx(64 * 10 / 2e-3)


def test_partition_balances_rows_and_covers_every_sequence():
    from linear_attention_serving_kda_gb300 import shard

    lens = np.array([6945, 2521, 1351, 2804, 3690, 6766, 3978, 1218, 0, 5])
    cu = np.concatenate([[0], np.cumsum(lens)])
    for world in (1, 2, 3, 4, 8, 16):
        parts = shard.partition_sequences(cu, world)
        assert len(parts) == world
        flat = sorted(s for p in parts for s in p)
        assert flat == list(range(len(lens)))          # every sequence exactly once
        loads = [int(lens[p].sum()) if p else 0 for p in parts]
        # greedy longest-first: no rank exceeds the best possible by more than the longest sequence
        assert max(loads) <= max(lens.sum() / world, lens.max()) + lens.max()
        assert parts == shard.partition_sequences(cu, world)  # deterministic
    with pytest.raises(ValueError):
        shard.partition_sequences([0, 5, 3], 2)


def test_prompt_cuts_cover_the_prompt_on_chunk_boundaries():
    from linear_attention_serving_kda_gb300 import shard

    for T in (0, 1, 63, 64, 65, 1000, 32768):
        for pieces in (1, 2, 3, 4, 7, 8):
            cuts = shard.prompt_cuts(T, pieces)
            assert len(cuts) <= pieces and (T > 0) == bool(cuts)
            assert [a for a, _ in cuts] == ([0] if T else []) + [b for _, b in cuts[:-1]]   # consecutive
            assert (cuts[-1][1] if cuts else 0) == T                                        # cover [0, T)
            assert all(a % 64 == 0 and a < b for a, b in cuts)
    with pytest.raises(ValueError):
        shard.prompt_cuts(10, 0)


def test_oracle_over_cuts_with_carried_states_is_the_uncut_run():
    """The oracle's serial recurrence run cut by cut, each cut starting from
    the previous cut's fp64 states, gives the uncut run bit for bit: the cuts
    move data only."""
    import oracle
    from linear_attention_serving_kda_gb300 import shard, workloads as W

    wl = W.make_workload("cuts", 43, [300], H=2, d=32, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    full = oracle.forward(wl, threads=1)
    outs, conv, rec = [], None, None
    for a, b in shard.prompt_cuts(wl.T, 3):
        sub = shard.cut_prompt(wl, a, b)
        arrays = dict(sub.arrays) if conv is None else dict(sub.arrays, conv_state=conv, rec_state=rec)
        res = oracle.forward(sub, threads=1, arrays=arrays)
        outs.append(res["out"])
        conv, rec = res["conv_state"], res["rec_state"]
    assert np.array_equal(np.concatenate(outs), full["out"])
    assert np.array_equal(rec, full["rec_state"]) and np.array_equal(conv, full["conv_state"])
    with pytest.raises(ValueError):
        shard.cut_prompt(W.make_workload("two", 1, [5, 6], H=1, d=16, K=4), 0, 3)


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from linear_attention_serving_kda_gb300 import shard, workloads as W

    wl = W.make_workload("dp", 41, [37, 130, 5, 64, 0, 71], H=2, d=32, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    seqs = shard.partition_sequences(wl.cu_seqlens, world)[rank]
    mine = oracle.forward(shard.shard_workload(wl, seqs), threads=1)
    got = [None] * world
    dist.all_gather_object(got, (seqs, mine))
    if rank == 0:
        full = oracle.forward(wl, threads=1)
        ok = True
        for sq, res in got:
            sub_cu = np.concatenate([[0], np.cumsum([wl.cu_seqlens[s + 1] - wl.cu_seqlens[s] for s in sq])]).astype(int)
            for j, s in enumerate(sq):
                a0, a1 = wl.cu_seqlens[s], wl.cu_seqlens[s + 1]
                ok &= np.array_equal(res["out"][sub_cu[j]:sub_cu[j + 1]], full["out"][a0:a1])
                ok &= np.array_equal(res["rec_state"][j], full["rec_state"][s])
                ok &= np.array_equal(res["conv_state"][j], full["conv_state"][s])
        out.put(bool(ok) and sorted(s for sq, _ in got for s in sq) == list(range(wl.N)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_sequences_bit_for_bit():
    """Two gloo ranks each run the oracle on their partition of a varlen
    batch; the gathered outputs and final states equal one unsharded run bit
    for bit (the units are independent: replicas need no data exchange)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
