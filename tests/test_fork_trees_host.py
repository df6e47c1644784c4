"""Fork-tree workloads (beam search, MCTS) on the host block manager (CPU only).

Repeated forks, frees and copy-on-write of shared tails: the C++ manager follows the
oracle op by op (slots, copy pairs, tables, free-list order, reference counts), and
the paging invariants of "PagedAttention: Virtual Memory Guide for LLM Inference"
("Key Architectural Mechanics" 1-2) hold after every op: a frame's reference count
is the number of tables holding it, free + held frames = all frames, and every
write lands in a frame only its writer holds.
"""

import pytest

import workloads
from oracle import OracleBlockManager

CASES = [
    ("beam", dict(n_prompts=3, prompt_len=50, width=4, steps=30, B=8)),
    ("beam", dict(n_prompts=2, prompt_len=17, width=8, steps=40, B=4)),
    ("beam", dict(n_prompts=4, prompt_len=33, width=2, steps=25, B=16)),
    ("mcts", dict(n_roots=2, prompt_len=40, iterations=20, B=8)),
    ("mcts", dict(n_roots=3, prompt_len=7, iterations=30, batch=6, rollout_max=40, max_nodes=20, B=4)),
]


def build(kind, kw):
    return workloads.beam_search(**kw) if kind == "beam" else workloads.mcts_tree(**kw)


def invariants(ob):
    held = {}
    for t in ob.tables.values():
        for f in t:
            held[f] = held.get(f, 0) + 1
    for f in range(ob.num_blocks):
        assert ob.refs[f] == held.get(f, 0)
    assert len(ob.free_list) + len(held) == ob.num_blocks
    assert all(ob.refs[f] == 0 for f in ob.free_list)


@pytest.mark.parametrize("kind,kw", CASES)
def test_fork_tree_bit_exact(pa, kind, kw):
    w = build(kind, kw)
    bm = pa.BlockManager(w.num_blocks, w.block_size, w.free_order)
    ob = OracleBlockManager(w.num_blocks, w.block_size, w.free_order)
    copies_seen = 0
    for op in w.ops:
        k = op[0]
        if k == "add":
            assert bm.add_seq(op[1], op[2]).tolist() == ob.add_seq(op[1], op[2])
        elif k == "fork":
            bm.fork(op[1], op[2])
            ob.fork(op[1], op[2])
        elif k == "free":
            assert bm.free(op[1]) == 0 and ob.free(op[1]) is None
        elif k in ("step", "extend"):
            got = bm.step(op[1]) if k == "step" else bm.extend(op[1], op[2])
            want = ob.step(list(op[1])) if k == "step" else ob.extend(op[1], op[2])
            assert got[0].tolist() == want[0]
            assert [tuple(c) for c in got[1].tolist()] == want[1]
            copies_seen += len(want[1])
            # each written slot's frame is held by its writer only
            seqs = list(op[1]) if k == "step" else [op[1]] * op[2]
            for s, slot in zip(seqs, want[0]):
                assert ob.refs[slot // w.block_size] == 1
        invariants(ob)
        assert bm.free_list() == list(ob.free_list) and bm.ref_counts() == ob.refs
    assert copies_seen > 0
    for s, t in ob.tables.items():
        assert bm.table(s) == t


def test_beam_search_keeps_width():
    w = workloads.beam_search(3, 20, 5, 12, B=8)
    live = {}
    for op in w.ops:
        if op[0] == "attend":
            assert len(op[1]) == 3 * 5


@pytest.mark.parametrize("kind,kw", [c for c in CASES if c[0] == "beam"])
def test_grouped_selection_equals_interleaved(pa, kind, kw):
    """A beam-search selection (the forks and frees between two steps) applied as one
    batched fork call and then one batched free call leaves the manager exactly as the
    interleaved single calls do: a fork copies a live beam's table and never touches
    the free list, and a freed beam is never forked from, so a free cannot release a
    frame a later fork copies.  Checked against the oracle's op-by-op replay."""
    w = build(kind, kw)
    ob = OracleBlockManager(w.num_blocks, w.block_size, list(w.free_order))
    bm = pa.BlockManager(w.num_blocks, w.block_size, w.free_order)
    ops = w.ops
    i = 0
    while i < len(ops):
        op = ops[i]
        if op[0] in ("fork", "free"):
            j = i
            while j < len(ops) and ops[j][0] in ("fork", "free"):
                j += 1
            for o in ops[i:j]:  # oracle: interleaved, one at a time
                if o[0] == "fork":
                    ob.fork(o[1], o[2])
                else:
                    ob.free(o[1])
            forks = [o for o in ops[i:j] if o[0] == "fork"]
            bm.fork_many([o[1] for o in forks], [o[2] for o in forks])
            bm.free_many([o[1] for o in ops[i:j] if o[0] == "free"])
            assert bm.free_list() == list(ob.free_list) and bm.ref_counts() == ob.refs
            for s_, t in ob.tables.items():
                assert bm.table(s_) == t
            i = j
            continue
        if op[0] == "add":
            assert bm.add_seq(op[1], op[2]).tolist() == ob.add_seq(op[1], op[2])
        elif op[0] == "step":
            slots, copies = bm.step(op[1])
            oslots, ocopies = ob.step(op[1])
            assert slots.tolist() == list(oslots)
            assert [tuple(c) for c in copies] == [tuple(c) for c in ocopies]
        i += 1
    invariants(ob)

