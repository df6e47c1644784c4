"""Oracle decode attention over a paged cache, in float64.

"Solving the LLM Memory Wall" ("1. The Mathematical Foundation"): for a query q
and the sequence's keys k_j and values v_j,
    a_j = (q . k_j) * scale,        o = sum_j softmax(a)_j v_j,
with scale = 1/sqrt(d) passed in by the caller (the float32 value the kernel
receives).  The paging changes only how k_j, v_j are fetched ("The difference
isn't in the math"): the sequence's frames are gathered in table order, flattened
to [n_frames*B, H, D] and trimmed to the context length ("Implementation",
PagedAttention.forward).  Reading: the newest token (appended this step) is part of
the attended set, i.e. the causal j <= i form with i the new token.

Several queries per sequence (prefill / chunked prefill): the general causal form
of the same equation, o_i = sum_{j <= i} softmax(a_ij) v_j -- query i attends the
keys at positions 0..i.  A chunk of n queries is the last n positions of the
sequence (its keys already written to the cache).

The split-context merge (partial softmax states combined with log-sum-exp) is
not on the pages; its definition is stated here so the merge kernel has an oracle:
for a token subset P, m_P = max a_j, l_P = sum e^{a_j - m_P},
o_P = sum e^{a_j - m_P} v_j (unnormalised); over disjoint subsets covering the
sequence, out = sum_P e^{m_P - M} o_P / sum_P e^{m_P - M} l_P with M = max m_P.
"""

from __future__ import annotations

import numpy as np

from .cache import decode_storage


def attention_fp64(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """q [H, D], K/V [L, H, D] (float64) -> out [H, D]; L == 0 gives zeros."""
    H, D = q.shape
    if K.shape[0] == 0:
        return np.zeros((H, D), np.float64)
    a = np.einsum("hd,lhd->hl", q, K) * float(scale)
    a -= a.max(axis=1, keepdims=True)
    w = np.exp(a)
    w /= w.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", w, V)


def gather(cache, table, L: int):
    """Frames of ``table`` concatenated in order, flattened and trimmed to L tokens."""
    B, H, D = cache.block_size, cache.num_heads, cache.head_dim
    n_frames = -(-L // B)
    if n_frames == 0:
        empty = np.zeros((0, H, D), np.float64)
        return empty, empty
    ks = np.concatenate([cache.frame("k", b) for b in table[:n_frames]], axis=0)[:L]
    vs = np.concatenate([cache.frame("v", b) for b in table[:n_frames]], axis=0)[:L]
    return decode_storage(ks, cache.dtype), decode_storage(vs, cache.dtype)


def paged_decode(q: np.ndarray, cache, tables, lens, scale: float) -> np.ndarray:
    """q [S, H, D] in storage dtype; tables[s] a frame list; lens[s] the context length."""
    qd = decode_storage(q, cache.dtype)
    out = np.zeros(qd.shape, np.float64)
    for s in range(qd.shape[0]):
        K, V = gather(cache, tables[s], int(lens[s]))
        out[s] = attention_fp64(qd[s], K, V, scale)
    return out


def paged_prefill(q: np.ndarray, cache, tables, lens, query_start, scale: float) -> np.ndarray:
    """Causal attention for chunks of queries.

    q [T, H, D] (storage dtype): rows query_start[s] .. query_start[s+1]-1 are the
    last n_s = query_start[s+1] - query_start[s] positions of sequence s (length
    lens[s]); row r at position p attends keys 0..p.  Returns float64 [T, H, D].
    """
    qd = decode_storage(q, cache.dtype)
    out = np.zeros(qd.shape, np.float64)
    for s in range(len(lens)):
        a, b = int(query_start[s]), int(query_start[s + 1])
        L = int(lens[s])
        K, V = gather(cache, tables[s], L)
        for r in range(a, b):
            pos = L - (b - a) + (r - a)
            out[r] = attention_fp64(qd[r], K[: pos + 1], V[: pos + 1], scale)
    return out


def prefill_weight_bound(q: np.ndarray, cache, tables, lens, query_start, scale: float) -> np.ndarray:
    """Per output element, sum_j w_j |v_j| (softmax weights times value magnitudes).

    A kernel that rounds the softmax weights to a u-precision type before the
    value product can be off by at most u * this (plus its own fp32 error)."""
    qd = decode_storage(q, cache.dtype)
    bound = np.zeros(qd.shape, np.float64)
    for s in range(len(lens)):
        a, b = int(query_start[s]), int(query_start[s + 1])
        L = int(lens[s])
        K, V = gather(cache, tables[s], L)
        for r in range(a, b):
            pos = L - (b - a) + (r - a)
            bound[r] = attention_fp64(qd[r], K[: pos + 1], np.abs(V[: pos + 1]), scale)
    return bound


def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """(m [H], l [H], o [H, D]) of one token subset, float64."""
    a = np.einsum("hd,lhd->hl", q, K) * float(scale)
    m = a.max(axis=1)
    e = np.exp(a - m[:, None])
    return m, e.sum(axis=1), np.einsum("hl,lhd->hd", e, V)


def lse_merge(parts):
    """Combine partial states [(m, l, o), ...] of disjoint token subsets."""
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    num = sum(np.exp(m - M)[:, None] * o for m, _, o in parts)
    den = sum(np.exp(m - M) * l for m, l, _ in parts)
    return num / den[:, None]


def round_to_storage(x: np.ndarray, dtype: str):
    """Round float64 values to the output dtype, nearest-even; returns float64 values."""
    x = np.asarray(x, np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # Via float32 (exact RNE), then float32 -> bf16 RNE; a float32 value that
        # lands exactly on a bf16 halfway point after the first rounding is
        # resolved by the sign of the first rounding's error (no double rounding).
        x32 = x.astype(np.float32)
        bits = x32.view(np.uint32).astype(np.uint64)
        low = bits & 0xFFFF
        hi = bits >> 16
        up = (low > 0x8000) | ((low == 0x8000) & ((hi & 1) == 1))
        tie_fix = (low == 0x8000) & (x32.astype(np.float64) != x)
        away = np.abs(x) > np.abs(x32.astype(np.float64))
        up = np.where(tie_fix, away, up)
        rb = (hi + up.astype(np.uint64)).astype(np.uint32) << np.uint32(16)
        return rb.view(np.float32).astype(np.float64)
    raise ValueError(dtype)
