"""Pins for the oracle's translation, cache model, attention and merge (CPU only).

References used, none of which is the oracle's own code path:
  * the address formula of "PagedAttention: Virtual Memory Guide for LLM
    Inference" ("The Mathematics of Block Translation"), checked against NumPy's
    own byte strides of an interleaved K/V frame buffer;
  * PyTorch's scaled_dot_product_attention (a different implementation) on a
    contiguous cache, i.e. an identity block table;
  * closed forms: one token gives v_0; equal keys give the mean of V; two tokens
    give the logistic mix; a constant shift of all values shifts the output;
  * brute force at 50 significant digits (mpmath) on tiny inputs;
  * exact bf16 rounding by enumerating neighbouring representable values.
"""

import math

import numpy as np
import pytest
import torch

from oracle import (
    OracleBlockManager,
    OracleKVCache,
    attention_fp64,
    decode_storage,
    lse_merge,
    paged_decode,
    partial_state,
    round_to_storage,
)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------- translation
@pytest.mark.parametrize("B,H,D,dt", [(10, 2, 64, np.float32), (16, 3, 8, np.float16), (4, 1, 4, np.float64)])
def test_address_formula_on_interleaved_frames(B, H, D, dt):
    """Address(K_i) = table[i//B]*FrameSize + (i mod B)*(2*H*D*bytes).

    The formula describes a frame holding K and V rows together, i.e. a buffer
    [num_blocks, B, 2, H, D]; its K_i is element [table[i//B], i mod B, 0, 0, 0].
    The oracle's slot (frame*B + offset) times the interleaved row size must equal
    the formula, and NumPy's byte offset of that element must equal both.
    """
    e = np.dtype(dt).itemsize
    nb = 12
    buf = np.zeros((nb, B, 2, H, D), dt)
    frame_size = B * 2 * H * D * e
    bm = OracleBlockManager(nb, B, free_order=list(np.random.default_rng(1).permutation(nb)))
    bm.add_seq(0, 3 * B + 1)
    for i in range(3 * B + 1):
        b, o = i // B, i % B
        addr = bm.tables[0][b] * frame_size + o * (2 * H * D * e)
        numpy_off = int(np.dot([bm.tables[0][b], o, 0, 0, 0], buf.strides))
        assert addr == numpy_off
        assert bm.slot(0, i) * (2 * H * D * e) == addr


def test_cache_write_lands_at_frame_and_offset():
    B, H, D = 10, 2, 4
    bm = OracleBlockManager(8, B, free_order=[5, 2, 7, 0, 1, 3, 4, 6])
    cache = OracleKVCache(8, B, H, D, "f32")
    slots = bm.add_seq(0, 23)
    k = _rand((23, H, D), 0).astype(np.float32)
    v = _rand((23, H, D), 1).astype(np.float32)
    cache.write(slots, k, v)
    for i in range(23):
        frame = bm.tables[0][i // B]
        assert np.array_equal(cache.k[frame, i % B], k[i])
        assert np.array_equal(cache.v[frame, i % B], v[i])
    untouched = [b for b in range(8) if b not in bm.tables[0]]
    assert not cache.k[untouched].any() and not cache.v[untouched].any()
    # tail slots of the last frame stay zero
    assert not cache.k[bm.tables[0][2], 3:].any()


# --------------------------------------------------------------------------- attention
def test_single_token_returns_its_value():
    q = _rand((3, 8), 0)
    K = _rand((1, 3, 8), 1)
    V = _rand((1, 3, 8), 2)
    assert np.array_equal(attention_fp64(q, K, V, 0.35), V[0])


def test_equal_keys_average_values():
    q = _rand((2, 8), 0)
    K = np.repeat(_rand((1, 2, 8), 1), 7, axis=0)
    V = _rand((7, 2, 8), 2)
    np.testing.assert_allclose(attention_fp64(q, K, V, 0.5), V.mean(axis=0), rtol=0, atol=1e-14)


def test_two_tokens_logistic_mix():
    q = _rand((1, 4), 3)
    K = _rand((2, 1, 4), 4)
    V = _rand((2, 1, 4), 5)
    scale = 0.7
    d = scale * (q[0] @ K[0, 0] - q[0] @ K[1, 0])
    w0 = 1.0 / (1.0 + math.exp(-d))
    np.testing.assert_allclose(attention_fp64(q, K, V, scale)[0], w0 * V[0, 0] + (1 - w0) * V[1, 0],
                               rtol=0, atol=1e-14)


def test_value_shift_and_linearity():
    q, K = _rand((2, 8), 6), _rand((9, 2, 8), 7)
    V1, V2 = _rand((9, 2, 8), 8), _rand((9, 2, 8), 9)
    c = _rand((2, 8), 10)
    o1 = attention_fp64(q, K, V1, 0.3)
    np.testing.assert_allclose(attention_fp64(q, K, V1 + c, 0.3), o1 + c, atol=1e-13)
    np.testing.assert_allclose(attention_fp64(q, K, V1 + V2, 0.3),
                               o1 + attention_fp64(q, K, V2, 0.3), atol=1e-13)


def test_empty_context_is_zero():
    assert not attention_fp64(_rand((2, 4), 0), np.zeros((0, 2, 4)), np.zeros((0, 2, 4)), 1.0).any()


def test_brute_force_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    q, K, V = _rand((2, 3), 11), _rand((5, 2, 3), 12), _rand((5, 2, 3), 13)
    scale = 0.57735
    got = attention_fp64(q, K, V, scale)
    for h in range(2):
        logits = [mpmath.mpf(scale) * sum(mpmath.mpf(q[h, d]) * mpmath.mpf(K[j, h, d]) for d in range(3))
                  for j in range(5)]
        den = sum(mpmath.e ** a for a in logits)
        for d in range(3):
            num = sum(mpmath.e ** logits[j] * mpmath.mpf(V[j, h, d]) for j in range(5))
            assert abs(float(num / den) - got[h, d]) < 1e-14


@pytest.mark.parametrize("L,B", [(1, 4), (7, 4), (16, 16), (17, 16), (45, 10)])
def test_identity_table_matches_torch_sdpa(L, B):
    """Identity block table == dense attention by a different implementation."""
    H, D = 3, 16
    nb = -(-L // B) + 2
    cache = OracleKVCache(nb, B, H, D, "f32")
    bm = OracleBlockManager(nb, B)            # free list 0.. -> identity table
    slots = bm.add_seq(0, L)
    assert bm.tables[0] == list(range(-(-L // B)))
    k = _rand((L, H, D), 20).astype(np.float32)
    v = _rand((L, H, D), 21).astype(np.float32)
    cache.write(slots, k, v)
    q = _rand((1, H, D), 22).astype(np.float32)
    scale = float(np.float32(1) / np.sqrt(np.float32(D)))
    got = paged_decode(q, cache, bm.tables, [L], scale)[0]
    tq = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]    # [1, H, 1, D]
    tk = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2)[None]    # [1, H, L, D]
    tv = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, :, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_physical_permutation_invariance_is_exact():
    H, D, B, L = 2, 8, 4, 27
    nb = 10
    outs = []
    for seed in range(4):
        order = list(np.random.default_rng(seed).permutation(nb))
        bm = OracleBlockManager(nb, B, free_order=order)
        cache = OracleKVCache(nb, B, H, D, "f16")
        slots = bm.add_seq(0, L)
        cache.write(slots, _rand((L, H, D), 1).astype(np.float16), _rand((L, H, D), 2).astype(np.float16))
        outs.append(paged_decode(_rand((1, H, D), 3).astype(np.float16), cache, bm.tables, [L], 0.25))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_bf16_storage_decodes_exactly():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F], np.uint16)
    want = [1.0, -1.0, 3.140625, 0.0, -0.0, 3.3895313892515355e38]
    assert decode_storage(bits, "bf16").tolist() == want


# --------------------------------------------------------------------------- merge
@pytest.mark.parametrize("cuts", [[5], [1, 2, 3], [10, 11], [3, 9, 14, 19]])
def test_lse_merge_equals_full_softmax(cuts):
    q, K, V = _rand((3, 8), 30), _rand((20, 3, 8), 31), _rand((20, 3, 8), 32)
    edges = [0] + cuts + [20]
    parts = [partial_state(q, K[a:b], V[a:b], 0.4) for a, b in zip(edges[:-1], edges[1:])]
    np.testing.assert_allclose(lse_merge(parts), attention_fp64(q, K, V, 0.4), rtol=0, atol=1e-13)


def test_lse_merge_two_single_tokens_closed_form():
    q, K, V = _rand((1, 4), 40), _rand((2, 1, 4), 41), _rand((2, 1, 4), 42)
    parts = [partial_state(q, K[i:i + 1], V[i:i + 1], 1.0) for i in range(2)]
    for m, l, o in parts:
        assert l[0] == 1.0                      # a single token's own weight is e^0
    d = q[0] @ K[0, 0] - q[0] @ K[1, 0]
    w0 = 1.0 / (1.0 + math.exp(-d))
    np.testing.assert_allclose(lse_merge(parts)[0], w0 * V[0, 0] + (1 - w0) * V[1, 0], atol=1e-14)


# --------------------------------------------------------------------------- rounding
def _bf16_nearest_even(x):
    """Brute force: nearest bf16 value by scanning neighbours, ties to even mantissa."""
    f = np.float32(x)
    base = int(f.view(np.uint32)) >> 16
    best = None
    for cand in (base - 1, base, base + 1, base + 2):
        val = float(np.uint32((cand & 0xFFFF) << 16).view(np.float32))
        key = (abs(val - x), cand & 1)
        if best is None or key < best[0]:
            best = (key, val)
    return best[1]


def test_round_to_bf16_nearest_even():
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(2000) * 3,
                         # float64 values just off bf16 midpoints (double-rounding traps)
                         np.array([1.0 + 2 ** -8 + 2 ** -30, 1.0 + 2 ** -8 - 2 ** -30, 1.0 + 2 ** -8,
                                   1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8 + 2 ** -40)])])
    got = round_to_storage(xs, "bf16")
    want = np.array([_bf16_nearest_even(x) for x in xs])
    assert np.array_equal(got, want)


def test_round_to_f16_nearest_even():
    xs = np.concatenate([np.random.default_rng(6).standard_normal(5000) * 4,
                         np.array([1.0 + 2 ** -11 + 2 ** -40, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11])])
    got = round_to_storage(xs, "f16")
    for x, g in zip(xs, got):
        h = np.float16(x)
        cands = [np.nextafter(h, np.float16(-np.inf)), h, np.nextafter(h, np.float16(np.inf))]
        best = min(cands, key=lambda c: (abs(float(c) - x), int(c.view(np.uint16)) & 1))
        assert g == float(best)


# ------------------------------------------------------------------ split cache layout
def test_split_layout_matches_the_printed_shapes():
    """[VM] "3. PagedAttention CUDA Kernel Execution" prints k_cache as
    [num_blocks, num_heads, head_dim/x, block_size, x] and v_cache as
    [num_blocks, num_heads, head_dim, block_size].  Row-major byte offsets of those
    shapes (closed form) locate, in the arrays split_layout returns, exactly the
    element k[f, b, h, d] (v[f, b, h, d]) of the [nb, B, H, D] caches."""
    import numpy as np

    from oracle import split_layout

    rng = np.random.default_rng(3)
    for dtype, e in ((np.float16, 2), (np.float32, 4)):
        nb, B, H, D = 5, 16, 3, 64
        x = 16 // e
        k = rng.standard_normal((nb, B, H, D)).astype(dtype)
        v = rng.standard_normal((nb, B, H, D)).astype(dtype)
        ks, vs = split_layout(k, v, e)
        assert ks.shape == (nb, H, D // x, B, x) and vs.shape == (nb, H, D, B)
        kb, vb = ks.tobytes(), vs.tobytes()
        for _ in range(200):
            f, b, h, d = (int(rng.integers(n)) for n in (nb, B, H, D))
            ko = ((((f * H + h) * (D // x) + d // x) * B + b) * x + d % x) * e
            vo = (((f * H + h) * D + d) * B + b) * e
            assert np.frombuffer(kb[ko:ko + e], dtype)[0] == k[f, b, h, d]
            assert np.frombuffer(vb[vo:vo + e], dtype)[0] == v[f, b, h, d]
