"""Oracle replay of the seeded workloads (CPU only).

The toy workload is the worked allocation trace of "PagedAttention, simply
explained"; its replay must reproduce the printed tables and free list.  The
scaled-down variants of the other workloads must keep the paging invariants and
give finite attention within the convex hull of the values.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import replay


def test_toy_replay_reproduces_worked_trace(golden):
    g = golden("worked_allocation_trace.json")
    w = workloads.build(0)
    res = replay(w, snapshots=True)
    step_ops = [i for i, op in enumerate(w.ops) if op[0] == "step"]
    last = res.snapshots[step_ops[-1]]
    names = g["order"]
    final = g["steps"][-1]
    assert {n: last["tables"][i] for i, n in enumerate(names)} == final["tables"]
    assert last["free"][:3] == final["free_head"] and len(last["free"]) == final["free_len"]
    # per-step slots of the hand derivation (frame*10 + offset)
    assert [res.trace[i]["slots"] for i in step_ops] == [[8, 15, 32, 49], [9, 16, 33, 50], [60, 17, 34, 51]]
    assert len(res.outputs) == 3
    for out in res.outputs.values():
        assert np.isfinite(out).all()


@pytest.mark.parametrize("cfg", [1, "1x", 2, 3, 4])
def test_small_workloads_replay(cfg):
    w = workloads.build(cfg, small=True)
    res = replay(w)
    bm = res.bm
    live = {}
    for s, t in bm.tables.items():
        assert len(t) == -(-bm.lens[s] // w.block_size)
        for b in t:
            live[b] = live.get(b, 0) + 1
    assert all(bm.refs[b] == c for b, c in live.items())
    assert len(bm.free_list) + len(live) == w.num_blocks
    (op_i,) = w.attend_ops[-1:]
    out = res.outputs[op_i]
    assert np.isfinite(out).all()
    # softmax output is a convex combination of the sequence's values
    tables, lens = res.attend_meta[op_i]
    from oracle.attention import gather
    for j, (t, L) in enumerate(zip(tables, lens)):
        _, V = gather(res.cache, t, L)
        assert (out[j] <= V.max(axis=0) + 1e-12).all() and (out[j] >= V.min(axis=0) - 1e-12).all()
    if cfg == 3:
        copies = sum(len(r["copies"]) for r in res.trace.values())
        assert copies > 0


def test_sampled_replay_matches_full_replay():
    w = workloads.build(3, small=True)
    full = replay(w)
    keep = [1, 5, 6]
    part = replay(w, keep_seqs=keep)
    op_i = w.attend_ops[-1]
    assert np.array_equal(full.outputs[op_i][keep], part.outputs[op_i][keep])


def test_generator_is_deterministic_and_rounds_like_torch():
    w1, w2 = workloads.build(4, small=True), workloads.build(4, small=True)
    k1, v1 = w1.rows(0)
    k2, v2 = w2.rows(0)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert np.array_equal(w1.free_order, w2.free_order)
    # bf16 bit patterns equal torch's float32 -> bfloat16 rounding of the same draws
    ss = np.random.SeedSequence([w1.seed, 0, 1])
    x = np.random.Generator(np.random.PCG64(ss)).standard_normal(k1.size, dtype=np.float32) * np.float32(0.5)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(k1.reshape(-1), ref)
