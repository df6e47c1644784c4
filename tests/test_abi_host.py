"""C-ABI library checks that need no GPU (CPU only).

* libpa.so loads and exports every function include/pa.h declares.
* The C++ host block manager matches the oracle block manager bit for bit:
  tables, lengths, free-list order, reference counts, slots and copy pairs, on
  the pages' traces and on seeded random operation sequences.
* Error behaviour: all-or-nothing steps and prompts, unknown / duplicate ids,
  double free, bad arguments.
"""

import json
import os
import random
import re
import subprocess

import numpy as np
import pytest

from oracle import DOUBLE_FREE, OracleBlockManager, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(pa):
    names = _declared()
    assert len(names) >= 20
    nm = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b[TW] (pa_[a-z0-9_]+)$", nm, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(pa.LIB, n)
    assert sorted(pa.EXPORTED) == names


def test_strerror_and_launch_count(pa):
    assert pa.pa_strerror(0) == "ok"
    assert "free blocks" in pa.pa_strerror(-6)
    assert pa.pa_launch_count() >= 0


# ------------------------------------------------------------------------------- parity
def _same_state(bm, ob):
    assert bm.num_free == ob.free_count
    assert bm.free_list() == list(ob.free_list)
    assert bm.ref_counts() == ob.refs
    assert bm.num_seqs == len(ob.tables)
    for s, t in ob.tables.items():
        assert bm.table(s) == t
        assert bm.seq_info(s) == (ob.lens[s], len(t))
    assert bm.usage() == ob.usage()
    ex = bm.export()
    assert ex["tables"] == ob.tables and ex["lens"] == ob.lens
    assert ex["free"] == list(ob.free_list) and ex["refs"] == ob.refs


def test_worked_trace_bit_exact(pa, golden):
    g = golden("worked_allocation_trace.json")
    bm = pa.BlockManager(g["num_blocks"], g["block_size"])
    ob = OracleBlockManager(g["num_blocks"], g["block_size"])
    for i, name in enumerate(g["order"]):
        assert bm.add_seq(i, g["prefill"][name]).tolist() == ob.add_seq(i, g["prefill"][name])
    _same_state(bm, ob)
    for _ in g["steps"]:
        slots, copies = bm.step([0, 1, 2, 3])
        oslots, ocopies = ob.step([0, 1, 2, 3])
        assert slots.tolist() == oslots and copies.tolist() == [list(c) for c in ocopies]
        _same_state(bm, ob)
    assert {n: bm.table(i) for i, n in enumerate(g["order"])} == g["steps"][-1]["tables"]


def test_cow_trace_bit_exact(pa, golden):
    g = golden("cow_trace.json")
    e = g["expect"]
    bm = pa.BlockManager(g["num_blocks"], g["block_size"])
    bm.add_seq(0, g["prompt"])
    bm.fork(0, 1)
    slot, cp = bm.append(0)
    assert slot == e["append_alpha"]["slot"] and list(cp) == e["append_alpha"]["copy"]
    assert bm.table(0) == e["append_alpha"]["alpha"] and bm.table(1) == e["append_alpha"]["beta"]
    slot, cp = bm.append(1)
    assert slot == e["append_beta"]["slot"] and cp is None
    bm.free(0)
    bm.free(1)
    assert bm.free_list()[-3:] == e["free_tail_after_both"]


@pytest.mark.parametrize("seed", range(10))
def test_random_ops_bit_exact(pa, seed):
    rnd = random.Random(1000 + seed)
    B = rnd.choice([1, 2, 4, 10, 16, 32])
    n = rnd.randint(8, 80)
    order = rnd.sample(range(n), n)
    bm = pa.BlockManager(n, B, order)
    ob = OracleBlockManager(n, B, order)
    next_id = 0
    for _ in range(500):
        r = rnd.random()
        live = list(ob.tables)
        if r < 0.2 or not live:
            L = rnd.randint(0, 3 * B)
            try:
                want = ob.add_seq(next_id, L)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as ei:
                    bm.add_seq(next_id, L)
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                assert bm.add_seq(next_id, L).tolist() == want
            next_id += 1
        elif r < 0.35:
            p = rnd.choice(live)
            ob.fork(p, next_id)
            bm.fork(p, next_id)
            next_id += 1
        elif r < 0.45:
            s = rnd.choice(live + [10 ** 6])
            want = ob.free(s)
            got = bm.free(s)
            assert (got == pa.PA_WARN_DOUBLE_FREE) == (want == DOUBLE_FREE)
        elif r < 0.55:
            s, n_new = rnd.choice(live), rnd.randint(0, 2 * B + 3)
            try:
                want = ob.extend(s, n_new)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as ei:
                    bm.extend(s, n_new)
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                slots, copies = bm.extend(s, n_new)
                assert slots.tolist() == want[0]
                assert [tuple(c) for c in copies.tolist()] == want[1]
        else:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 5))]  # repeats allowed
            try:
                want = ob.step(seqs)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as ei:
                    bm.step(seqs)
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                slots, copies = bm.step(seqs)
                assert slots.tolist() == want[0]
                assert [tuple(c) for c in copies.tolist()] == want[1]
        _same_state(bm, ob)
        for s in ob.tables:
            if ob.lens[s]:
                i = rnd.randrange(ob.lens[s])
                assert bm.slot(s, i) == ob.slot(s, i)


def test_block_tables_export(pa):
    bm = pa.BlockManager(16, 4, list(range(15, -1, -1)))
    bm.add_seq(7, 9)
    bm.add_seq(3, 0)
    tables, lens = bm.block_tables([7, 3], 5)
    assert tables.tolist() == [[15, 14, 13, -1, -1], [-1] * 5]
    assert lens.tolist() == [9, 0]
    with pytest.raises(pa.PAError):
        bm.block_tables([7], 2)                 # table longer than max_blocks


def test_errors_leave_state_unchanged(pa):
    bm = pa.BlockManager(3, 2)
    bm.add_seq(0, 2)
    bm.add_seq(1, 2)
    before = (bm.free_list(), bm.ref_counts(), bm.table(0), bm.table(1))
    with pytest.raises(pa.PAError) as ei:
        bm.step([0, 1])                         # second spill has no frame left
    assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
    assert (bm.free_list(), bm.ref_counts(), bm.table(0), bm.table(1)) == before
    with pytest.raises(pa.PAError) as ei:
        bm.step([0, 99])
    assert ei.value.code == pa.PA_ERR_UNKNOWN_SEQ
    assert (bm.free_list(), bm.ref_counts(), bm.table(0), bm.table(1)) == before
    with pytest.raises(pa.PAError) as ei:
        bm.add_seq(0, 1)
    assert ei.value.code == pa.PA_ERR_SEQ_EXISTS
    with pytest.raises(pa.PAError):
        bm.add_seq(5, 7)                        # needs 4 frames, 1 free
    assert (bm.free_list(), bm.ref_counts()) == before[:2]
    with pytest.raises(pa.PAError):
        bm.fork(42, 43)
    with pytest.raises(pa.PAError):
        pa.BlockManager(4, 2, [0, 1, 1, 2])     # not a permutation
    with pytest.raises(pa.PAError):
        pa.BlockManager(0, 2)
    assert bm.free(0) == 0
    assert bm.free(0) == pa.PA_WARN_DOUBLE_FREE


@pytest.mark.parametrize("seed", range(4))
def test_batched_fork_and_free_match_the_oracle(pa, seed):
    """fork_many / free_many = the same forks / frees one at a time (oracle), including
    chained forks inside one batch; a bad batch changes nothing."""
    rnd = random.Random(seed)
    n, B = 64, 4
    order = rnd.sample(range(n), n)
    bm = pa.BlockManager(n, B, order)
    ob = OracleBlockManager(n, B, order)
    for s in range(4):
        L = rnd.randint(1, 9)
        assert bm.add_seq(s, L).tolist() == ob.add_seq(s, L)
    nid = 100
    for _ in range(12):
        live = sorted(ob.tables)
        parents, children = [], []
        for _ in range(rnd.randint(1, 5)):
            parents.append(rnd.choice(live + children))
            children.append(nid)
            nid += 1
        bm.fork_many(parents, children)
        for p_, c_ in zip(parents, children):
            ob.fork(p_, c_)
        step = rnd.sample(sorted(ob.tables), min(3, len(ob.tables)))
        slots, copies = bm.step(step)
        oslots, ocopies = ob.step(step)
        assert slots.tolist() == list(oslots) and [tuple(c) for c in copies] == [tuple(c) for c in ocopies]
        dead = rnd.sample(sorted(ob.tables), max(0, len(ob.tables) - 6))
        assert bm.free_many(dead) == 0
        for d in dead:
            ob.free(d)
        assert bm.free_list() == list(ob.free_list) and bm.ref_counts() == ob.refs
        for s_, t in ob.tables.items():
            assert bm.table(s_) == t
    live = sorted(ob.tables)
    before = (bm.free_list(), bm.ref_counts(), [bm.table(s_) for s_ in live])
    with pytest.raises(pa.PAError) as ei:
        bm.fork_many([live[0], 999999], [nid, nid + 1])        # second parent unknown
    assert ei.value.code == pa.PA_ERR_UNKNOWN_SEQ
    with pytest.raises(pa.PAError) as ei:
        bm.fork_many([live[0], live[0]], [nid, nid])           # child twice
    assert ei.value.code == pa.PA_ERR_SEQ_EXISTS
    with pytest.raises(pa.PAError) as ei:
        bm.fork_many([live[0]], [live[1]])                     # child already live
    assert ei.value.code == pa.PA_ERR_SEQ_EXISTS
    with pytest.raises(pa.PAError) as ei:
        bm.fork_many([nid + 1, live[0]], [nid, nid + 1])       # parent born only later in the batch
    assert ei.value.code == pa.PA_ERR_UNKNOWN_SEQ
    assert (bm.free_list(), bm.ref_counts(), [bm.table(s_) for s_ in live]) == before
    assert bm.free_many([live[0], live[0]]) == pa.PA_WARN_DOUBLE_FREE  # second is not live
    assert bm.free_many([]) == 0


def test_engine_picks_the_shared_prefix_path(pa):
    """The engine decodes through the shared-prefix path exactly when two neighbouring
    sequences of the batch start on the same frame (and never overrides the caller)."""
    import types

    pick = pa.PagedKVEngine._decode_params
    on, off = types.SimpleNamespace(auto_share=True), types.SimpleNamespace(auto_share=False)
    forked = np.array([[5, 9, 2], [5, 9, 7], [1, 3, -1]], np.int32)
    apart = np.array([[5, 9, 2], [6, 9, 7], [5, 3, -1]], np.int32)   # equal first frames, not neighbours
    empty = np.array([[-1, -1], [-1, -1]], np.int32)
    assert pick(on, forked, None) == {"share_prefix": 1}
    assert pick(on, apart, None) is None
    assert pick(on, empty, None) is None
    assert pick(on, forked[:1], None) is None
    assert pick(off, forked, None) is None
    assert pick(on, forked, {}) == {}
    assert pick(on, forked, {"partition_tokens": -1}) == {"partition_tokens": -1}


# ------------------------------------------------------------------ prefix caching
from oracle.prefix_cache import OraclePrefixBlockManager  # noqa: E402


def _same_cache_state(bm, ob):
    _same_state(bm, ob)
    assert bm.cached_frames() == ob.cached_frames()


def test_prefix_cache_trace_bit_exact(pa, golden):
    g = golden("prefix_cache_trace.json")
    bm = pa.BlockManager(g["num_blocks"], g["block_size"])
    ob = OraclePrefixBlockManager(g["num_blocks"], g["block_size"])
    for st in g["steps"]:
        exp = st["expect"]
        if st["op"] == "add_cached":
            if exp.get("error") == "out_of_blocks":
                with pytest.raises(pa.PAError) as ei:
                    bm.add_seq_cached(st["seq"], st["tokens"])
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
                with pytest.raises(OutOfBlocks):
                    ob.add_seq_cached(st["seq"], st["tokens"])
            else:
                n_cached, slots = bm.add_seq_cached(st["seq"], st["tokens"])
                assert n_cached == exp["n_cached"] and slots.tolist() == exp["slots"]
                ob.add_seq_cached(st["seq"], st["tokens"])
        elif st["op"] == "free":
            assert bm.free(st["seq"]) == 0
            ob.free(st["seq"])
        elif st["op"] == "extend":
            slots, copies = bm.extend_tokens(st["seq"], st["tokens"])
            assert slots.tolist() == exp["slots"] and copies.tolist() == exp["copies"]
            ob.extend(st["seq"], len(st["tokens"]), st["tokens"])
        if "free" in exp:
            assert bm.free_list() == exp["free"]
        if "cached" in exp:
            assert bm.cached_frames() == exp["cached"]
        _same_cache_state(bm, ob)


@pytest.mark.parametrize("seed", range(12))
def test_prefix_cache_random_ops_bit_exact(pa, seed):
    rnd = random.Random(7000 + seed)
    B = rnd.choice([1, 2, 4, 8, 16])
    n = rnd.randint(10, 70)
    order = rnd.sample(range(n), n)
    bm = pa.BlockManager(n, B, order)
    ob = OraclePrefixBlockManager(n, B, order)
    prompts = [[rnd.randint(0, 3) for _ in range(rnd.randint(0, 5 * B))] for _ in range(4)]
    next_id, hits = 0, 0
    for _ in range(400):
        live = list(ob.tables)
        r = rnd.random()
        if r < 0.3 or not live:
            base = rnd.choice(prompts)
            cut = rnd.randint(0, len(base))
            toks = base[:cut] + [rnd.randint(0, 3) for _ in range(rnd.randint(0, 3 * B))]
            try:
                want = ob.add_seq_cached(next_id, toks)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as ei:
                    bm.add_seq_cached(next_id, toks)
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                got = bm.add_seq_cached(next_id, toks)
                assert got[0] == want[0] and got[1].tolist() == want[1]
                hits += want[0]
                if rnd.random() < 0.3:
                    prompts.append(toks)
            next_id += 1
        elif r < 0.35:
            L = rnd.randint(0, 2 * B)               # a prompt without token ids
            try:
                want = ob.add_seq(next_id, L)
            except OutOfBlocks:
                with pytest.raises(pa.PAError):
                    bm.add_seq(next_id, L)
            else:
                assert bm.add_seq(next_id, L).tolist() == want
            next_id += 1
        elif r < 0.45:
            p = rnd.choice(live)
            ob.fork(p, next_id)
            bm.fork(p, next_id)
            next_id += 1
        elif r < 0.6:
            s = rnd.choice(live)
            assert (bm.free(s) == pa.PA_WARN_DOUBLE_FREE) == (ob.free(s) is not None)
        else:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 4))]
            with_tokens = rnd.random() < 0.8
            toks = [rnd.randint(0, 3) for _ in seqs]
            single = rnd.random() < 0.3
            try:
                if single:
                    want = ob.extend(seqs[0], len(seqs), toks if with_tokens else None)
                else:
                    want = ob.step(seqs, toks if with_tokens else None)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as ei:
                    if single:
                        bm.extend_tokens(seqs[0], toks) if with_tokens else bm.extend(seqs[0], len(seqs))
                    else:
                        bm.step_tokens(seqs, toks) if with_tokens else bm.step(seqs)
                assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                if single:
                    got = bm.extend_tokens(seqs[0], toks) if with_tokens else bm.extend(seqs[0], len(seqs))
                else:
                    got = bm.step_tokens(seqs, toks) if with_tokens else bm.step(seqs)
                assert got[0].tolist() == want[0]
                assert [tuple(c) for c in got[1].tolist()] == want[1]
        _same_cache_state(bm, ob)
    assert hits >= 0


def test_prefix_cache_errors(pa):
    bm = pa.BlockManager(4, 2)
    assert bm.add_seq_cached(0, [1, 2, 3])[0] == 0
    with pytest.raises(pa.PAError) as ei:
        bm.add_seq_cached(0, [1, 2])
    assert ei.value.code == pa.PA_ERR_SEQ_EXISTS
    before = (bm.free_list(), bm.ref_counts(), bm.cached_frames())
    with pytest.raises(pa.PAError) as ei:
        bm.add_seq_cached(1, [9] * 7)                      # 4 new frames, 2 free
    assert ei.value.code == pa.PA_ERR_OUT_OF_BLOCKS
    assert (bm.free_list(), bm.ref_counts(), bm.cached_frames()) == before
    n_cached, slots = bm.add_seq_cached(2, [])             # empty prompt: nothing to look up
    assert n_cached == 0 and len(slots) == 0
    with pytest.raises(ValueError):
        bm.step_tokens([0, 2], [5])                        # one token id per sequence


def test_memory_report_lines(pa, capsys):
    # bench.py --memory: one line per workload from the native manager's accounting;
    # every sequence wastes fewer than B slots, and at B = 16 the paged waste stays
    # under the pages' 4 % on every realistic workload.
    import bench
    bench.memory_report()
    lines = [json.loads(x) for x in capsys.readouterr().out.splitlines() if x.startswith("{")]
    assert [x["key"] for x in lines] == ["0", "1", "1x", "2", "3", "4", "beam", "prefix"]
    for x in lines:
        assert 0 <= x["max_seq_waste_slots"] <= x["waste_bound_slots"] == x["block_size"] - 1
        assert x["slots_filled"] <= x["slots_allocated"] == x["frames_in_use"] * x["block_size"]
        if x["block_size"] == 16:
            assert x["paged_waste_pct"] < 4.0
    shared = {x["key"]: x["shared_frames_saving_pct"] for x in lines}
    assert shared["3"] > 50 and shared["beam"] > 50 and shared["prefix"] > 50 and shared["1"] == 0


def test_cpu_baseline_worker_runs():
    # The oracle timing behind bench.py's cpu_baseline and --cpu-sweep (toy workload).
    import bench
    r = bench.cpu_baseline_worker(0, 0.2, seed_shift=3)
    assert r["kind"] == "oracle" and r["cores"] == 1
    assert r["value"] > 0 and r["seqs_per_sec"] > 0


def test_every_error_code_has_a_message(pa):
    # each PA_ERR_* / PA_WARN_* code the header defines has its own message
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")).read()
    codes = {name: int(v) for name, v in re.findall(r"#define (PA_(?:ERR|WARN)_\w+)\s+(-?\d+)", text)}
    assert "PA_ERR_HOST_MEMORY" in codes
    unknown = pa.pa_strerror(-999)
    msgs = {name: pa.pa_strerror(v) for name, v in codes.items()}
    assert all(m and m != unknown for m in msgs.values()), msgs
    assert len(set(msgs.values())) == len(msgs)
    assert getattr(pa, "PA_ERR_HOST_MEMORY") == codes["PA_ERR_HOST_MEMORY"]


def test_export_capacity_and_arguments(pa):
    import ctypes as C
    import numpy as np
    bm = pa.BlockManager(10, 4)
    bm.add_seq(7, 9)
    bm.add_seq(3, 2)
    assert bm.export() == {"tables": {3: [3], 7: [0, 1, 2]}, "lens": {3: 2, 7: 9},
                           "free": [4, 5, 6, 7, 8, 9], "refs": [1, 1, 1, 1] + [0] * 6}
    lib = pa._binding.LIB
    ids, lens, offs = np.zeros(2, np.int64), np.zeros(2, np.int32), np.zeros(3, np.int64)
    tabs, free, refs = np.zeros(4, np.int32), np.zeros(10, np.int32), np.zeros(10, np.int32)
    ns, ne, nf = C.c_int32(), C.c_int64(), C.c_int32()
    i64 = lambda a: a.ctypes.data_as(C.POINTER(C.c_int64))
    i32 = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))
    args = lambda cs, ce: (bm.handle, i64(ids), i32(lens), i64(offs), i32(tabs), i32(free), i32(refs), cs, ce,
                           C.byref(ns), C.byref(ne), C.byref(nf))
    assert lib.pa_bm_export(*args(1, 4)) == pa.PA_ERR_CAPACITY            # two sequences live
    assert (ns.value, ne.value, nf.value) == (2, 4, 6)
    assert lib.pa_bm_export(*args(2, 3)) == pa.PA_ERR_CAPACITY            # four table entries
    assert lib.pa_bm_export(*args(2, 4)) == 0
    assert ids.tolist() == [3, 7] and offs.tolist() == [0, 1, 4] and tabs.tolist() == [3, 0, 1, 2]
    assert lib.pa_bm_export(*args(-1, 4)) == pa._binding.PA_ERR_INVALID
    bm.close()
