"""Pins for the oracle's causal multi-query (prefill / chunked-prefill) attention (CPU).

References: the oracle's decode attention (itself pinned) for one query per
sequence; PyTorch's scaled_dot_product_attention with an explicit causal mask
(a different implementation) on contiguous frames; 50-digit brute force; and the
weight bound's defining identity.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import (
    OracleBlockManager,
    OracleKVCache,
    paged_decode,
    paged_prefill,
    prefill_weight_bound,
    replay,
)


def _contiguous(L, H, D, B, seed, dtype="f32"):
    nb = -(-L // B) + 1
    bm = OracleBlockManager(nb, B)
    cache = OracleKVCache(nb, B, H, D, dtype)
    slots = bm.add_seq(0, L)
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, H, D)).astype(np.float32)
    v = rng.standard_normal((L, H, D)).astype(np.float32)
    cache.write(slots, k, v)
    return bm, cache, k, v


@pytest.mark.parametrize("L,n,B", [(1, 1, 4), (9, 9, 4), (40, 7, 16), (37, 37, 10), (100, 33, 16)])
def test_matches_torch_sdpa_with_causal_mask(L, n, B):
    H, D = 3, 16
    bm, cache, k, v = _contiguous(L, H, D, B, seed=L + n)
    q = np.random.default_rng(5).standard_normal((n, H, D)).astype(np.float32)
    scale = 0.25
    got = paged_prefill(q, cache, bm.tables, [L], [0, n], scale)
    pos = np.arange(L - n, L)
    mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])          # [n, L] True = attend
    tq = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_full_prefill_is_torch_is_causal():
    H, D, L, B = 2, 8, 50, 16
    bm, cache, k, v = _contiguous(L, H, D, B, seed=3)
    q = np.random.default_rng(4).standard_normal((L, H, D)).astype(np.float32)
    got = paged_prefill(q, cache, bm.tables, [L], [0, L], 0.3)
    t = lambda x: torch.from_numpy(x.astype(np.float64)).permute(1, 0, 2)[None]  # noqa: E731
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=0.3)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_single_query_chunk_equals_decode():
    w = workloads.build(1, small=True)
    res = replay(w)
    op = w.attend_ops[-1]
    tables, lens = res.attend_meta[op]
    q = w.query(op)
    S = len(lens)
    got = paged_prefill(q, res.cache, tables, lens, list(range(S + 1)), w.scale)
    assert np.array_equal(got, paged_decode(q, res.cache, tables, lens, w.scale))


def test_brute_force_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    H, D, L, n, B = 1, 3, 5, 3, 2
    bm, cache, k, v = _contiguous(L, H, D, B, seed=9)
    q = np.random.default_rng(10).standard_normal((n, H, D)).astype(np.float32)
    got = paged_prefill(q, cache, bm.tables, [L], [0, n], 0.7)
    for i in range(n):
        pos = L - n + i
        logits = [mpmath.mpf(0.7) * sum(mpmath.mpf(float(q[i, 0, d])) * mpmath.mpf(float(k[j, 0, d]))
                                        for d in range(D)) for j in range(pos + 1)]
        den = sum(mpmath.e ** x for x in logits)
        for d in range(D):
            num = sum(mpmath.e ** logits[j] * mpmath.mpf(float(v[j, 0, d])) for j in range(pos + 1))
            assert abs(float(num / den) - got[i, 0, d]) < 1e-14


def test_weight_bound_identity():
    H, D, L, B = 2, 8, 30, 16
    bm, cache, k, v = _contiguous(L, H, D, B, seed=12)
    q = np.random.default_rng(13).standard_normal((6, H, D)).astype(np.float32)
    bound = prefill_weight_bound(q, cache, bm.tables, [L], [0, 6], 0.2)
    out = paged_prefill(q, cache, bm.tables, [L], [0, 6], 0.2)
    assert (bound >= np.abs(out) - 1e-12).all()
    # with non-negative values the bound is the output itself
    cache.v[:] = np.abs(cache.v)
    np.testing.assert_allclose(prefill_weight_bound(q, cache, bm.tables, [L], [0, 6], 0.2),
                               paged_prefill(q, cache, bm.tables, [L], [0, 6], 0.2), rtol=0, atol=1e-13)


def test_extend_is_repeated_append():
    a, b = OracleBlockManager(20, 4), OracleBlockManager(20, 4)
    a.add_seq(0, 6)
    b.add_seq(0, 6)
    slots, copies = a.extend(0, 9)
    want = [b.append(0)[0] for _ in range(9)]
    assert slots == want and copies == [] and a.snapshot() == b.snapshot()


def test_chunked_prefill_workload_replays():
    w = workloads.prefill_batch(small=True)
    res = replay(w)
    (op,) = w.prefill_ops
    out = res.outputs[op]
    assert out.shape[0] == sum(w.ops[op][2]) and np.isfinite(out).all()


def test_off_by_one_causal_bound_is_caught(monkeypatch):
    import oracle.attention as att
    orig = att.attention_fp64

    def shifted(q, K, V, scale):      # attends one key too few
        return orig(q, K[:-1], V[:-1], scale) if K.shape[0] > 1 else orig(q, K, V, scale)
    monkeypatch.setattr(att, "attention_fp64", shifted)
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa_with_causal_mask(40, 7, 16)
