"""Pins for the prefix-caching oracle (CPU only).

* a hand-derived trace (tests/golden/prefix_cache_trace.json): hits, revival of a
  freed cached frame, eviction when a cached frame is handed out again, a miss after
  eviction, all-or-nothing admission, registration by token appends;
* the defining property of prefix reuse, on seeded random operation sequences: the
  contents every live sequence reads through its table are exactly what its own
  token prefix produces (a content model in which a slot stores the identity of the
  token prefix written there);
* without token ids the manager behaves exactly like the base block manager;
* planted mistakes (a key without its parent, a revived frame left in the free
  list, an evicted key kept, the last token allowed to hit) each break a pin.
"""

import random

import pytest

from oracle import OracleBlockManager, OutOfBlocks
from oracle.prefix_cache import OraclePrefixBlockManager


def _check_expect(bm, seq, exp, got=None):
    if "table" in exp:
        assert bm.tables[seq] == exp["table"]
    if "free" in exp:
        assert list(bm.free_list) == exp["free"]
    if "refs" in exp:
        assert bm.refs == exp["refs"]
    if "cached" in exp:
        assert bm.cached_frames() == exp["cached"]


def replay_trace(bm, g):
    for st in g["steps"]:
        exp = st["expect"]
        if st["op"] == "add_cached":
            if exp.get("error") == "out_of_blocks":
                with pytest.raises(OutOfBlocks):
                    bm.add_seq_cached(st["seq"], st["tokens"])
            else:
                n_cached, slots = bm.add_seq_cached(st["seq"], st["tokens"])
                assert n_cached == exp["n_cached"] and slots == exp["slots"]
        elif st["op"] == "free":
            assert bm.free(st["seq"]) is None
        elif st["op"] == "extend":
            slots, copies = bm.extend(st["seq"], len(st["tokens"]), st["tokens"])
            assert slots == exp["slots"] and [list(c) for c in copies] == exp["copies"]
        _check_expect(bm, st.get("seq"), exp)
    fin = g["final"]
    assert {str(s): t for s, t in bm.tables.items()} == fin["tables"]
    assert {str(s): n for s, n in bm.lens.items()} == fin["lens"]
    assert list(bm.free_list) == fin["free"] and bm.refs == fin["refs"] and bm.cached_frames() == fin["cached"]


def test_hand_derived_trace(golden):
    g = golden("prefix_cache_trace.json")
    replay_trace(OraclePrefixBlockManager(g["num_blocks"], g["block_size"]), g)


# ------------------------------------------------------------------ content model
class ContentModel:
    """Each slot holds the identity of the token prefix whose K/V was written there
    (a real model's K/V row of token j depends on tokens 0..j)."""

    def __init__(self, num_blocks, B):
        self.slots = [None] * (num_blocks * B)
        self.B = B

    def write(self, slots, prefixes):
        for s, p in zip(slots, prefixes):
            self.slots[s] = p

    def copy_block(self, src, dst):
        B = self.B
        self.slots[dst * B:(dst + 1) * B] = self.slots[src * B:(src + 1) * B]


def prefix_ids(tokens, start, stop):
    return [tuple(tokens[:j + 1]) for j in range(start, stop)]


def check_contents(bm, cm):
    for s, table in bm.tables.items():
        toks = bm.tokens[s]
        for j in range(bm.lens[s]):
            if toks[j] is None:
                continue
            if any(t is None for t in toks[:j + 1]):
                continue
            assert cm.slots[bm.slot(s, j)] == tuple(toks[:j + 1]), (s, j)
    # a registered frame holds the block of its key's content
    for node, frame in bm.node_frame.items():
        assert bm.frame_node[frame] == node
    for f, node in enumerate(bm.frame_node):
        if node:
            assert bm.node_frame[node] == f


def _random_tokens(rnd, prompts, L):
    base = rnd.choice(prompts)
    cut = rnd.randint(0, len(base))
    return base[:cut] + [rnd.randint(0, 3) for _ in range(L - cut)]


def run_random(bm_cls, seed, ops=400, planted=None):
    rnd = random.Random(seed)
    B = rnd.choice([1, 2, 4, 8])
    n = rnd.randint(12, 60)
    order = rnd.sample(range(n), n)
    bm = bm_cls(n, B, order)
    if planted:
        planted(bm)
    cm = ContentModel(n, B)
    prompts = [[rnd.randint(0, 3) for _ in range(rnd.randint(0, 5 * B))] for _ in range(4)]
    next_id = 0
    hits = 0
    for _ in range(ops):
        r = rnd.random()
        live = list(bm.tables)
        if r < 0.35 or not live:
            toks = _random_tokens(rnd, prompts, rnd.randint(0, 5 * B))
            try:
                n_cached, slots = bm.add_seq_cached(next_id, toks)
            except OutOfBlocks:
                pass
            else:
                hits += n_cached
                assert n_cached % B == 0 and n_cached <= max(0, len(toks) - 1)
                cm.write(slots, prefix_ids(toks, n_cached, len(toks)))
                if rnd.random() < 0.3:
                    prompts.append(list(toks))
            next_id += 1
        elif r < 0.45:
            p = rnd.choice(live)
            bm.fork(p, next_id)
            next_id += 1
        elif r < 0.65:
            bm.free(rnd.choice(live))
        else:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 3))]
            toks = [rnd.randint(0, 3) for _ in seqs]
            before = {s: list(bm.tokens[s]) for s in set(seqs)}
            try:
                slots, copies = bm.step(seqs, toks)
            except OutOfBlocks:
                continue
            for src, dst in copies:      # copies come before the step's writes
                cm.copy_block(src, dst)
            cur = dict(before)
            for s, t, slot in zip(seqs, toks, slots):
                cur[s] = cur[s] + [t]
                cm.write([slot], [tuple(cur[s])] if None not in cur[s] else [None])
        check_contents(bm, cm)
        live_frames = {f for t in bm.tables.values() for f in t}
        assert len(bm.free_list) + len(live_frames) == bm.num_blocks
        assert len(set(bm.free_list)) == len(bm.free_list)
        assert all(bm.refs[f] == 0 for f in bm.free_list)
    return hits


@pytest.mark.parametrize("seed", range(12))
def test_reused_frames_hold_the_sequence_prefix(seed):
    assert run_random(OraclePrefixBlockManager, seed) >= 0


def test_random_runs_do_hit():
    assert sum(run_random(OraclePrefixBlockManager, s) for s in range(12)) > 0


@pytest.mark.parametrize("seed", range(6))
def test_without_tokens_same_as_base_manager(seed):
    rnd = random.Random(seed)
    B = rnd.choice([1, 2, 4, 10, 16])
    n = rnd.randint(8, 64)
    order = rnd.sample(range(n), n)
    a, b = OracleBlockManager(n, B, order), OraclePrefixBlockManager(n, B, order)
    nid = 0
    for _ in range(300):
        live = list(a.tables)
        r = rnd.random()
        if r < 0.25 or not live:
            L = rnd.randint(0, 3 * B)
            res = []
            for m in (a, b):
                try:
                    res.append(m.add_seq(nid, L))
                except OutOfBlocks:
                    res.append("oob")
            assert res[0] == res[1]
            nid += 1
        elif r < 0.4:
            p = rnd.choice(live)
            a.fork(p, nid)
            b.fork(p, nid)
            nid += 1
        elif r < 0.55:
            s = rnd.choice(live)
            assert a.free(s) == b.free(s)
        else:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 4))]
            res = []
            for m in (a, b):
                try:
                    res.append(m.step(seqs))
                except OutOfBlocks:
                    res.append("oob")
            assert res[0] == res[1]
        assert a.snapshot()["tables"] == b.snapshot()["tables"]
        assert list(a.free_list) == list(b.free_list) and a.refs == b.refs
        assert not any(b.cached_frames())


# ------------------------------------------------------------------ planted mistakes
class KeyWithoutParent(OraclePrefixBlockManager):
    def _key(self, parent, toks):
        return (0, tuple(toks))


class RevivedLeftInFreeList(OraclePrefixBlockManager):
    def _revive(self, frame):
        self.refs[frame] += 1


class EvictionKeepsKey(OraclePrefixBlockManager):
    def _evict(self, node):
        self.frame_node[self.node_frame[node]] = 0


class LastTokenMayHit(OraclePrefixBlockManager):
    def _hit_limit(self, L):
        return L


def _fails(cls):
    for s in range(40):
        try:
            run_random(cls, s, ops=250)
        except (AssertionError, KeyError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("cls", [KeyWithoutParent, RevivedLeftInFreeList, EvictionKeepsKey])
def test_planted_mistakes_are_caught(cls):
    assert _fails(cls)


def test_planted_last_token_hit_is_caught(golden):
    g = golden("prefix_cache_trace.json")
    with pytest.raises(AssertionError):
        replay_trace(LastTokenMayHit(g["num_blocks"], g["block_size"]), g)


# ------------------------------------------------------------------ attention through reused frames
def _logical_prefill(w, op_index, seq_pos, seq, count):
    """Definition: causal attention over the sequence's own token rows (no cache,
    no block table), for its last `count` positions."""
    import numpy as np

    from oracle import attention_fp64, decode_storage

    toks = w.token_history(op_index)[seq]
    L = len(toks)
    k, v = w.prefix_rows(toks)
    K, V = decode_storage(k, w.dtype), decode_storage(v, w.dtype)
    q = decode_storage(w.position_queries(op_index)[seq_pos][L - count:], w.dtype)
    return np.stack([attention_fp64(q[r], K[:L - count + r + 1], V[:L - count + r + 1], w.scale)
                     for r in range(count)])


@pytest.mark.parametrize("turns,free_between,B", [(1, False, 8), (2, False, 8), (3, True, 4), (2, False, 16)])
def test_prefill_through_reused_frames_equals_definition(turns, free_between, B):
    import numpy as np

    import workloads
    from oracle import replay

    w = workloads.shared_prefix(3, 37, [11, 20, 4], B=B, turns=turns, reply_len=7, free_between=free_between,
                                seed=30 + turns)
    r = replay(w)
    assert sum(r.n_cached.values()) > 0          # the workload does reuse blocks
    for i in w.prefill_ops + [j for j, op in enumerate(w.ops) if op[0] == "prefill_new"]:
        if w.ops[i][0] != "prefill_new":
            continue
        tables, lens, counts = r.attend_meta[i]
        for j, s in enumerate(w.ops[i][1]):
            want = _logical_prefill(w, i, j, s, counts[j])
            np.testing.assert_allclose(r.outputs[i][j], want, rtol=0, atol=1e-12)


def test_usage_counts_cached_free_frames():
    # A freed prompt's filled blocks stay registered while free; a prompt that reuses
    # one takes it off the free list (no longer counted as cached-and-free), the
    # partial block was never registered.
    B = 4
    bm = OraclePrefixBlockManager(10, B)
    first = list(range(100, 110))  # 10 tokens: blocks 0, 1 filled, block 2 partial
    bm.add_seq_cached(0, first)
    u = bm.usage()
    assert (u["frames_in_use"], u["frames_cached"], u["slots_filled"]) == (3, 0, 10)
    bm.free(0)
    u = bm.usage()
    assert (u["frames_in_use"], u["frames_cached"], u["num_seqs"]) == (0, 2, 0)
    n_cached, _ = bm.add_seq_cached(1, first[:4] + [7, 7])  # block 0 hits, block 1 is new
    assert n_cached == 4
    u = bm.usage()
    assert (u["frames_in_use"], u["frames_cached"], u["slots_filled"]) == (2, 1, 6)
