"""Data-parallel replicas: which sequences each rank prefills.

The layer's (sequence, head) units never exchange data, so N GPUs run N
independent replicas, each over its own sequences (one process per GPU,
weak scaling, no collective on the data path).  This module holds the host
side of that split: a balanced assignment of whole sequences to ranks by row
count, and the pure data movement that cuts a rank's shard out of a batch
(rows, initial states).  No arithmetic of the layer is here.
"""
from __future__ import annotations

import numpy as np


def partition_sequences(cu_seqlens, world: int):
    """Assign whole sequences to `world` ranks, balancing row counts: longest
    first, each to the rank with the fewest rows so far (ties: lowest rank;
    equal lengths: lowest sequence index first).  Returns one ascending list
    of sequence indices per rank.  Deterministic, so every rank computes the
    same split from the same cu_seqlens without communicating."""
    if world < 1:
        raise ValueError("world must be >= 1")
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    if np.any(lens < 0):
        raise ValueError("cu_seqlens must be non-decreasing")
    order = sorted(range(len(lens)), key=lambda s: (-int(lens[s]), s))
    load = [0] * world
    parts = [[] for _ in range(world)]
    for s in order:
        r = min(range(world), key=lambda i: (load[i], i))
        parts[r].append(s)
        load[r] += int(lens[s])
    return [sorted(p) for p in parts]


def shard_workload(wl, seqs):
    """The sub-batch of a workload holding sequences `seqs` (in that order):
    their rows, their initial conv and recurrent states, the same parameters.
    Pure data movement."""
    from . import workloads as W

    cu = wl.cu_seqlens
    idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if len(seqs) else np.zeros(0, np.int64)
    lens = [int(cu[s + 1] - cu[s]) for s in seqs]
    sub = W.Workload(**{**wl.__dict__, "arrays": {}})
    sub.name = f"{wl.name}[{len(seqs)} seqs]"
    sub.cu_seqlens = np.zeros(len(lens) + 1, dtype=np.int32)
    sub.cu_seqlens[1:] = np.cumsum(lens)
    sel = np.asarray(seqs, dtype=np.int64)
    for nm, a in wl.arrays.items():
        if nm in ("q", "k", "v", "f", "b", "g"):
            sub.arrays[nm] = np.ascontiguousarray(a[idx])
        elif nm in ("conv_state", "rec_state", "accepted"):
            sub.arrays[nm] = np.ascontiguousarray(a[sel])
        else:
            sub.arrays[nm] = a
    return sub


def cut_prompt(wl, start: int, stop: int):
    """Rows [start, stop) of a one-sequence workload as a one-sequence
    workload of its own (same parameters and initial states).  Run in order
    with the states carried from one cut to the next, cuts at multiples of
    the 64-row chunk give the uncut prompt's result.  Pure data movement."""
    from . import workloads as W

    if wl.N != 1 or not 0 <= start <= stop <= wl.T:
        raise ValueError("cut_prompt wants one sequence and 0 <= start <= stop <= T")
    sub = W.Workload(**{**wl.__dict__, "arrays": {}})
    sub.name = f"{wl.name}[{start}:{stop}]"
    sub.cu_seqlens = np.array([0, stop - start], dtype=np.int32)
    for nm, a in wl.arrays.items():
        sub.arrays[nm] = np.ascontiguousarray(a[start:stop]) if nm in ("q", "k", "v", "f", "b", "g") else a
    return sub


def prompt_cuts(T: int, pieces: int, chunk: int = 64):
    """`pieces` (or fewer) consecutive (start, stop) row ranges covering
    [0, T), every boundary a multiple of `chunk`."""
    if pieces < 1:
        raise ValueError("pieces must be >= 1")
    step = max((T // pieces + chunk - 1) // chunk * chunk, chunk)
    return [(a, min(a + step, T)) for a in range(0, T, step)]
