"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case patches one plausible bug into the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong end of the free list, a missing
reference drop) and checks that at least one pin test then fails.  The patches
touch only the oracle, on the CPU.
"""

import numpy as np

import oracle.attention as att
import oracle.block_manager as bmmod
import tests.test_oracle_attention as TA
import tests.test_oracle_block_manager as TB


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _load(name):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


def test_swapped_k_and_v_is_caught(monkeypatch):
    orig = att.attention_fp64
    monkeypatch.setattr(att, "attention_fp64", lambda q, K, V, s: orig(q, V, K, s))
    monkeypatch.setattr(TA, "attention_fp64", att.attention_fp64)
    assert _fails(TA.test_single_token_returns_its_value)


def test_dropped_scale_is_caught(monkeypatch):
    orig = att.attention_fp64
    monkeypatch.setattr(att, "attention_fp64", lambda q, K, V, s: orig(q, K, V, 1.0))
    assert _fails(TA.test_identity_table_matches_torch_sdpa, 17, 16)


def test_wrong_softmax_sign_is_caught(monkeypatch):
    orig = att.attention_fp64
    monkeypatch.setattr(att, "attention_fp64", lambda q, K, V, s: orig(q, K, V, -s))
    monkeypatch.setattr(TA, "attention_fp64", att.attention_fp64)
    assert _fails(TA.test_two_tokens_logistic_mix)


def test_untrimmed_gather_is_caught(monkeypatch):
    def bad_gather(cache, table, L):
        B = cache.block_size
        n = -(-L // B)
        ks = np.concatenate([cache.frame("k", b) for b in table[:n]])
        vs = np.concatenate([cache.frame("v", b) for b in table[:n]])
        return att.decode_storage(ks, cache.dtype), att.decode_storage(vs, cache.dtype)
    monkeypatch.setattr(att, "gather", bad_gather)
    assert _fails(TA.test_identity_table_matches_torch_sdpa, 17, 16)


def test_merge_without_rescale_is_caught(monkeypatch):
    def bad_merge(parts):
        num = sum(o for _, _, o in parts)
        den = sum(l for _, l, _ in parts)
        return num / den[:, None]
    monkeypatch.setattr(TA, "lse_merge", bad_merge)
    assert _fails(TA.test_lse_merge_equals_full_softmax, [5])


def test_free_list_popped_from_back_is_caught(monkeypatch):
    def bad_take(self):
        frame = self.free_list.pop()
        self.refs[frame] = 1
        return frame
    monkeypatch.setattr(bmmod.OracleBlockManager, "_take_frame", bad_take)
    assert _fails(TB.test_worked_allocation_trace, _load)


def test_cow_without_reference_drop_is_caught(monkeypatch):
    monkeypatch.setattr(bmmod.OracleBlockManager, "_drop_ref", lambda self, f: None)
    assert _fails(TB.test_cow_trace, _load)


def test_offset_from_wrong_index_is_caught(monkeypatch):
    def bad_slot(self, seq, i):
        table = self.tables[seq]
        return table[i // self.block_size] * self.block_size + (i + 1) % self.block_size
    monkeypatch.setattr(bmmod.OracleBlockManager, "slot", bad_slot)
    assert _fails(TB.test_worked_trace_slots_hand_derived)


def test_freed_frames_to_front_is_caught(monkeypatch):
    def bad_drop(self, frame):
        if self.refs[frame] <= 0:
            return
        self.refs[frame] -= 1
        if self.refs[frame] == 0:
            self.free_list.appendleft(frame)
    monkeypatch.setattr(bmmod.OracleBlockManager, "_drop_ref", bad_drop)
    assert _fails(TB.test_fork_demo, _load)


def test_cow_copy_skipped_is_caught(monkeypatch):
    def bad_append(self, seq):
        t = self.lens[seq]
        table = self.tables[seq]
        if t % self.block_size == 0:
            table.append(self._take_frame())
        self.lens[seq] = t + 1
        return self.slot(seq, t), None
    monkeypatch.setattr(bmmod.OracleBlockManager, "append", bad_append)
    assert _fails(TB.test_cow_trace, _load)
