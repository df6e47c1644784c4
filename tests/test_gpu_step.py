"""GPU parity of the native decode step (pa_step_decode through PagedKVEngine.decode_step).

Workloads are replayed with every decode step and the attention that follows it fused
into one decode_step call (block-manager step, tables staged in pinned memory,
copy-on-write copies, append, decode in libpa).  Slots, copies, tables, reference counts and every
cache bit must equal the oracle's, attention outputs be within 2e-3 of it, and the
native path must give the same bits as the same step through the separate calls.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import replay
from tests._gpu_common import assert_attention_close, cache_bits, oracle_bits

pytestmark = pytest.mark.gpu


def replay_fused(pa, w, native=True, params=None):
    eng = pa.PagedKVEngine(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype,
                           free_order=w.free_order, max_seqs=max(64, len(w.final_lens)),
                           max_blocks_per_seq=max(1, max(-(-L // w.block_size) for L in w.final_lens.values())))
    dev = eng.device
    outs, ncs = {}, {}
    ops = w.ops
    i = 0
    while i < len(ops):
        op = ops[i]
        kind = op[0]
        if kind == "step" and i + 1 < len(ops) and ops[i + 1][0] == "attend" and tuple(ops[i + 1][1]) == tuple(op[1]):
            k, v = w.rows(i)
            kd, vd = pa.to_device_rows(k, w.dtype, dev), pa.to_device_rows(v, w.dtype, dev)
            q = pa.to_device_rows(w.query(i + 1), w.dtype, dev)
            ev = None if native else [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            out, nc, lens = eng.decode_step(op[1], kd, vd, q, w.scale, params=params, events=ev)
            outs[i + 1] = out.clone()
            ncs[i] = nc
            i += 2
            continue
        if kind == "add":
            k, v = w.rows(i)
            eng.add_seq(op[1], k, v)
        elif kind == "fork":
            eng.fork(op[1], op[2])
        elif kind == "free":
            eng.free(op[1])
        elif kind == "step":
            k, v = w.rows(i)
            eng.step(op[1], k, v)
        elif kind == "attend":
            outs[i] = eng.attend(op[1], w.query(i), w.scale, params=params).clone()
        else:
            raise ValueError(kind)
        i += 1
    torch.cuda.synchronize()
    return eng, outs, ncs


CASES = [
    ("decode batch", lambda: workloads.build(1, small=True)),
    # many steps without copy-on-write: the append reads its slots from the pinned ring and
    # carries the tables to the device itself; the ring (4 slots) wraps several times and
    # the batch changes size every other step
    ("decode steps", lambda: workloads.decode_steps([1, 15, 16, 17, 200, 31, 600, 2], 14, H=4, B=16,
                                                    dtype="f16", seed=74, drop_every=3)),
    ("decode steps bf16 B=8", lambda: workloads.decode_steps([7, 8, 9, 100, 64], 11, H=2, B=8, dtype="bf16",
                                                             seed=75, drop_every=2)),
    ("decode steps f32 D=64 B=10", lambda: workloads.decode_steps([3, 10, 11, 95, 40], 9, H=3, D=64, B=10,
                                                                 dtype="f32", seed=77, drop_every=2)),
    # 4 sequences for three steps, then all 420: the staged block outgrows the ring's
    # 16384 int32 per slot (420 x (4 + 46 table entries)) and the ring is reallocated
    # between steps
    ("decode steps, ring growth", lambda: workloads.decode_steps(
        [700 + (s * 37) % 31 for s in range(420)], 6, H=2, D=64, B=16, dtype="f16", seed=76, small_first=4)),
    ("beam search wide", lambda: workloads.beam_search(2, 150, 8, 16, H=4, B=16, dtype="f16", seed=73)),
    ("beam search", lambda: workloads.beam_search(3, 200, 4, 20, H=4, B=16, dtype="f16", seed=71)),
    ("beam search bf16 B=8", lambda: workloads.beam_search(2, 100, 8, 12, H=4, B=8, dtype="bf16", seed=72)),
    # 320 beams: the first decode step copies 316 shared tail frames, more than one launch's
    # parameters carry (256 pairs), so that step uploads its pairs; the later steps copy
    # 109 and 123 frames with the pairs in the launch parameters
    ("beam search, 316 copies in one step", lambda: workloads.beam_search(4, 30, 80, 4, H=2, B=16, dtype="f16",
                                                                         seed=78)),
    # the boundary of the copies carried in the launch parameters: 256 (the most that fit)
    # and 257 (uploaded) in the first step
    ("beam search, 256 copies in one step", lambda: workloads.beam_search(1, 20, 257, 2, H=2, B=16, dtype="f16",
                                                                         seed=79)),
    ("beam search, 257 copies in one step", lambda: workloads.beam_search(1, 20, 258, 2, H=2, B=16, dtype="bf16",
                                                                         seed=80)),
]


@pytest.mark.parametrize("name,make", CASES)
def test_native_step_matches_oracle_and_separate_calls(pa, name, make):
    w = make()
    eng, outs, ncs = replay_fused(pa, w, native=True)
    assert ncs, "the workload has no fused step"
    assert pa.pa_get_device_status() == 0
    ref = replay(w)
    assert eng.bm.free_list() == list(ref.bm.free_list)
    assert eng.bm.ref_counts() == ref.bm.refs
    for s, tab in ref.bm.tables.items():
        assert eng.bm.table(s) == tab
    assert np.array_equal(cache_bits(eng.k_cache), oracle_bits(ref.cache.k))
    assert np.array_equal(cache_bits(eng.v_cache), oracle_bits(ref.cache.v))
    for i, nc in ncs.items():
        assert nc == len(ref.trace[i]["copies"])
    assert outs
    for i, out in outs.items():
        assert_attention_close(out, ref.outputs[i], w.dtype)
    # the same replay through the separate calls gives the same bits
    eng2, outs2, _ = replay_fused(pa, w, native=False)
    for i in outs:
        assert torch.equal(outs[i].view(torch.int16), outs2[i].view(torch.int16)), i


def test_native_step_errors(pa):
    eng = pa.PagedKVEngine(8, 16, 4, 128, "f16", max_seqs=4, max_blocks_per_seq=2)
    eng.bm.add_seq(0, 31)
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    rows = torch.zeros_like(q)
    with pytest.raises(pa.PAError):          # unknown sequence: nothing changes
        eng.decode_step([5], rows, rows, q, 0.1)
    assert eng.bm.seq_info(0) == (31, 2)
    eng.decode_step([0], rows, rows, q, 0.1)  # 32 tokens: still 2 frames
    with pytest.raises(pa.PAError):          # 33 tokens need a third frame: more than max_blocks
        eng.decode_step([0], rows, rows, q, 0.1)
    before = eng.bm.seq_info(0)              # the capacity error's block-manager step stands
    with pytest.raises(ValueError):          # host rows: refused before anything runs
        eng.decode_step([0], rows.cpu(), rows, q, 0.1)
    assert eng.bm.seq_info(0) == before
    torch.cuda.synchronize()
