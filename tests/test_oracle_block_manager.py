"""Pins for the oracle block manager (CPU only).

Each test checks the oracle against something it does not compute itself: the
worked allocation trace printed in "PagedAttention, simply explained", the fork
demo of "PagedAttention: Virtual Memory Guide for LLM Inference", the slot
efficiency example of "Solving the LLM Memory Wall", a hand-derived copy-on-write
trace, and invariants that any correct paging state satisfies.
"""

import random

import pytest

from oracle import DOUBLE_FREE, OracleBlockManager, OutOfBlocks, SequenceExists, UnknownSequence


def _fill(bm, name_to_seq, fill):
    for name, expected in fill.items():
        s = name_to_seq[name]
        got = [[b, n] for b, n in zip(bm.tables[s], bm.fill_levels(s))]
        assert got == expected, name


def _free_matches(bm, head, last, length):
    fl = list(bm.free_list)
    assert fl[: len(head)] == head
    assert fl[-1] == last
    assert len(fl) == length


def test_worked_allocation_trace(golden):
    g = golden("worked_allocation_trace.json")
    bm = OracleBlockManager(g["num_blocks"], g["block_size"])
    seq = {name: i for i, name in enumerate(g["order"])}
    for name in g["order"]:
        bm.add_seq(seq[name], g["prefill"][name])
    ap = g["after_prefill"]
    _fill(bm, seq, ap["fill"])
    assert {n: bm.tables[seq[n]] for n in g["order"]} == ap["tables"]
    _free_matches(bm, ap["free_head"], ap["free_last"], ap["free_len"])
    for st in g["steps"]:
        bm.step([seq[n] for n in g["order"]])
        _fill(bm, seq, st["fill"])
        if "tables" in st:
            assert {n: bm.tables[seq[n]] for n in g["order"]} == st["tables"]
            _free_matches(bm, st["free_head"], st["free_last"], st["free_len"])
    # waste per request stays below one block (at most block_size - 1 slots)
    for s in seq.values():
        waste = len(bm.tables[s]) * bm.block_size - bm.lens[s]
        assert 0 <= waste <= bm.block_size - 1


def test_worked_trace_slots_hand_derived():
    # Slots implied by the printed tables and the translation frame*B + i mod B.
    bm = OracleBlockManager(100, 10)
    assert bm.add_seq(0, 8) == list(range(0, 8))
    assert bm.add_seq(1, 5) == list(range(10, 15))
    assert bm.add_seq(2, 12) == list(range(20, 32))
    assert bm.add_seq(3, 9) == list(range(40, 49))
    assert bm.step([0, 1, 2, 3]) == ([8, 15, 32, 49], [])
    assert bm.step([0, 1, 2, 3]) == ([9, 16, 33, 50], [])
    assert bm.step([0, 1, 2, 3]) == ([60, 17, 34, 51], [])
    assert [bm.lens[s] for s in range(4)] == [11, 8, 15, 12]
    assert [len(bm.tables[s]) * 10 - bm.lens[s] for s in range(4)] == [9, 2, 5, 8]


def test_fork_demo(golden):
    g = golden("fork_demo.json")
    bm = OracleBlockManager(g["num_blocks"], g["block_size"])
    a, b = 0, 1
    bm.add_seq(a, g["prompt"])
    assert bm.tables[a] == g["after_init"]["alpha"]
    assert bm.free_count == g["after_init"]["free_count"]
    bm.fork(a, b)
    assert bm.tables[b] == g["after_fork"]["beta"]
    assert bm.free_count == g["after_fork"]["free_count"]
    assert {str(k): bm.refs[k] for k in (0, 1)} == g["after_fork"]["refs"]
    slot, cp = bm.append(a)
    assert cp is None                        # boundary append: no copy
    assert slot == 2 * 16 + 0
    assert bm.tables[a] == g["after_append_alpha"]["alpha"]
    assert bm.tables[b] == g["after_append_alpha"]["beta"]
    assert bm.free_count == g["after_append_alpha"]["free_count"]
    bm.free(a)
    bm.free(b)
    assert bm.free_count == g["after_free_both"]["free_count"]
    assert list(bm.free_list)[-3:] == g["after_free_both"]["derived_free_tail"]


def test_cow_trace(golden):
    g = golden("cow_trace.json")
    e = g["expect"]
    bm = OracleBlockManager(g["num_blocks"], g["block_size"])
    bm.add_seq(0, g["prompt"])
    assert bm.tables[0] == e["alpha_after_add"]
    bm.fork(0, 1)
    slot, cp = bm.append(0)
    ea = e["append_alpha"]
    assert slot == ea["slot"] and list(cp) == ea["copy"]
    assert bm.tables[0] == ea["alpha"] and bm.tables[1] == ea["beta"]
    assert {str(k): bm.refs[k] for k in (0, 1, 2)} == ea["refs"]
    assert bm.free_count == ea["free_count"]
    slot, cp = bm.append(1)
    assert slot == e["append_beta"]["slot"] and cp is None
    assert bm.tables[1] == e["append_beta"]["beta"]
    assert bm.free_count == e["append_beta"]["free_count"]
    slot, cp = bm.append(1)
    assert slot == e["append_beta_2"]["slot"] and cp is None
    bm.free(0)
    bm.free(1)
    assert list(bm.free_list)[-3:] == e["free_tail_after_both"]
    assert bm.free_count == e["free_count_final"]


def test_slot_efficiency_example(golden):
    g = golden("slot_efficiency.json")
    bm = OracleBlockManager(16, g["block_size"])
    bm.add_seq(0, g["seq_len"])
    n_blocks = len(bm.tables[0])
    assert n_blocks == g["blocks"]
    assert n_blocks * g["block_size"] == g["slots"]
    assert n_blocks * g["block_size"] - g["seq_len"] == g["wasted_slots"]
    assert round(100 * g["seq_len"] / (n_blocks * g["block_size"]), 1) == g["efficiency_pct_approx"]
    assert round(100 * g["seq_len"] / g["contiguous_prealloc_slots"], 1) == g["contiguous_efficiency_pct_approx"]


def test_empty_prompt_takes_frame_on_first_append():
    bm = OracleBlockManager(4, 8)
    assert bm.add_seq(0, 0) == []
    assert bm.tables[0] == []
    assert bm.append(0) == (0, None)
    assert bm.tables[0] == [0]


def test_add_is_all_or_nothing():
    bm = OracleBlockManager(5, 4, free_order=[4, 3, 2, 1, 0])
    bm.add_seq(0, 12)                      # 3 frames: 4, 3, 2
    before = bm.snapshot()
    with pytest.raises(OutOfBlocks):
        bm.add_seq(1, 9)                   # needs 3, only 2 free
    assert bm.snapshot() == before
    with pytest.raises(SequenceExists):
        bm.add_seq(0, 1)


def test_step_is_all_or_nothing():
    bm = OracleBlockManager(3, 2)
    bm.add_seq(0, 2)                       # frame 0, full
    bm.add_seq(1, 2)                       # frame 1, full
    before = bm.snapshot()
    with pytest.raises(OutOfBlocks):
        bm.step([0, 1])                    # both spill, one frame left
    assert bm.snapshot() == before
    with pytest.raises(UnknownSequence):
        bm.step([0, 7])
    assert bm.snapshot() == before


def test_double_free_is_noop():
    bm = OracleBlockManager(4, 4)
    bm.add_seq(0, 5)
    assert bm.free(0) is None
    snap = bm.snapshot()
    assert bm.free(0) == DOUBLE_FREE
    assert bm.snapshot() == snap


def _check_invariants(bm):
    live = {}
    for s, table in bm.tables.items():
        assert len(table) == -(-bm.lens[s] // bm.block_size)
        waste = len(table) * bm.block_size - bm.lens[s]
        assert 0 <= waste < bm.block_size or (bm.lens[s] == 0 and waste == 0)
        for b in table:
            live[b] = live.get(b, 0) + 1
    for b in range(bm.num_blocks):
        assert bm.refs[b] == live.get(b, 0)
    assert set(bm.free_list).isdisjoint(live)
    assert len(bm.free_list) + len(live) == bm.num_blocks
    assert len(set(bm.free_list)) == len(bm.free_list)


@pytest.mark.parametrize("seed", range(6))
def test_random_ops_keep_invariants(seed):
    rnd = random.Random(seed)
    B = rnd.choice([1, 3, 4, 10, 16])
    n = rnd.randint(20, 60)
    bm = OracleBlockManager(n, B, free_order=rnd.sample(range(n), n))
    next_id = 0
    for _ in range(400):
        r = rnd.random()
        try:
            if r < 0.2 or not bm.tables:
                bm.add_seq(next_id, rnd.randint(0, 3 * B))
                next_id += 1
            elif r < 0.35:
                bm.fork(rnd.choice(list(bm.tables)), next_id)
                next_id += 1
            elif r < 0.45:
                bm.free(rnd.choice(list(bm.tables)))
            else:
                seqs = rnd.sample(list(bm.tables), k=min(len(bm.tables), rnd.randint(1, 4)))
                slots, copies = bm.step(seqs)
                # every slot lands in the writer's own, unshared tail frame
                for s, slot in zip(seqs, slots):
                    assert slot // B == bm.tables[s][(bm.lens[s] - 1) // B]
                    assert bm.refs[slot // B] == 1
                assert len(set(slots)) == len(slots)
                for src, dst in copies:
                    assert bm.refs[dst] == 1 and src != dst
        except OutOfBlocks:
            pass
        _check_invariants(bm)


# -- memory accounting (usage) ---------------------------------------------------------------

def test_usage_worked_trace(golden):
    # Final state of the printed trace: the fill levels it prints give the filled slots,
    # the frames and each request's waste ("max wastage per block is block_size minus 1").
    g = golden("worked_allocation_trace.json")
    bm = OracleBlockManager(g["num_blocks"], g["block_size"])
    seq = {name: i for i, name in enumerate(g["order"])}
    for name in g["order"]:
        bm.add_seq(seq[name], g["prefill"][name])
    for _ in g["steps"]:
        bm.step([seq[n] for n in g["order"]])
    fill = g["steps"][-1]["fill"]
    u = bm.usage()
    assert u["num_seqs"] == len(g["order"])
    assert u["frames_total"] == g["num_blocks"]
    assert u["frames_in_use"] == sum(len(v) for v in fill.values()) == u["table_entries"]
    assert u["slots_filled"] == sum(n for v in fill.values() for _, n in v) == u["tokens_logical"]
    assert u["max_seq_waste"] == max(len(v) * g["block_size"] - sum(n for _, n in v) for v in fill.values())
    assert u["max_seq_waste"] <= g["block_size"] - 1
    assert u["frames_cached"] == 0


def test_usage_slot_efficiency_example(golden):
    # "Performance Analysis": 7 tokens at B = 4 fill 7 of 8 slots (87.5 %), against 7 of a
    # 2048-slot contiguous reservation (0.3 %).
    g = golden("slot_efficiency.json")
    bm = OracleBlockManager(16, g["block_size"])
    bm.add_seq(0, g["seq_len"])
    u = bm.usage()
    assert u["frames_in_use"] * g["block_size"] == g["slots"]
    assert u["frames_in_use"] * g["block_size"] - u["slots_filled"] == g["wasted_slots"] == u["max_seq_waste"]
    assert round(100 * u["slots_filled"] / (u["frames_in_use"] * g["block_size"]), 1) == g["efficiency_pct_approx"]
    assert round(100 * u["tokens_logical"] / g["contiguous_prealloc_slots"], 1) == g["contiguous_efficiency_pct_approx"]


def test_usage_copy_on_write_trace(golden):
    # The hand-derived copy-on-write trace: after the fork both sequences hold frames 0, 1
    # once (2 frames for 4 table entries); alpha's write moves it to frame 2 (slot 36 =
    # frame 2, offset 4, so frame 2 holds 5 tokens) while beta keeps 4 tokens in frame 1;
    # beta's two in-place writes (slots 20, 21) bring frame 1 to 6.
    g = golden("cow_trace.json")
    B = g["block_size"]
    bm = OracleBlockManager(g["num_blocks"], B)
    bm.add_seq(0, g["prompt"])
    bm.fork(0, 1)
    u = bm.usage()
    assert (u["frames_in_use"], u["table_entries"]) == (2, 4)
    assert (u["slots_filled"], u["tokens_logical"]) == (g["prompt"], 2 * g["prompt"])
    slot, _ = bm.append(0)
    assert slot == g["expect"]["append_alpha"]["slot"]
    u = bm.usage()
    assert (u["frames_in_use"], u["table_entries"]) == (3, 4)
    assert u["slots_filled"] == B + (g["prompt"] - B) + (slot % B + 1)
    bm.append(1)
    bm.append(1)
    u = bm.usage()
    assert u["slots_filled"] == B + (g["prompt"] - B + 2) + (slot % B + 1)
    assert u["tokens_logical"] == 3 * g["prompt"] + 3 - g["prompt"]
    assert u["max_seq_waste"] == max(2 * B - (g["prompt"] + 1), 2 * B - (g["prompt"] + 2))


@pytest.mark.parametrize("seed", range(6))
def test_usage_brute_force(seed):
    # Filled slots = the distinct flat slots of every live (sequence, position); frames in
    # use = the distinct frames of the live tables; waste per sequence stays below B.
    rnd = random.Random(300 + seed)
    B = rnd.choice([1, 3, 8, 16])
    bm = OracleBlockManager(rnd.randint(20, 60), B)
    nxt = 0
    for _ in range(200):
        live = list(bm.tables)
        r = rnd.random()
        try:
            if r < 0.25 or not live:
                bm.add_seq(nxt, rnd.randint(0, 3 * B))
                nxt += 1
            elif r < 0.45:
                bm.fork(rnd.choice(live), nxt)
                nxt += 1
            elif r < 0.55:
                bm.free(rnd.choice(live))
            else:
                bm.step([rnd.choice(live) for _ in range(rnd.randint(1, 4))])
        except OutOfBlocks:
            pass
        u = bm.usage()
        slots = {bm.slot(s, i) for s in bm.tables for i in range(bm.lens[s])}
        frames = {f for t in bm.tables.values() for f in t}
        assert u["slots_filled"] == len(slots)
        assert u["frames_in_use"] == len(frames) == sum(1 for c in bm.refs if c > 0)
        assert u["table_entries"] == sum(len(t) for t in bm.tables.values())
        assert u["tokens_logical"] == sum(bm.lens.values())
        assert 0 <= u["max_seq_waste"] < B
        assert u["frames_in_use"] + bm.free_count == bm.num_blocks
