"""Helpers for the GPU parity tests: replay a workload through the CUDA path and the
oracle independently, then compare."""

from __future__ import annotations

import numpy as np
import torch

from oracle import replay, round_to_storage

TOL = 2e-3  # max abs error of attention outputs vs the fp64 oracle (fp32 accumulation)


def cache_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a device cache as a host array."""
    if t.dtype == torch.float32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_bits(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float32:
        return a.view(np.uint32)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    return a  # bf16 already as uint16 bits


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, dtype: str, tol: float = TOL) -> float:
    """|gpu - oracle| <= tol + |round(oracle) - oracle| element-wise.

    The second term is the rounding of the exact result to the output dtype,
    which no kernel can avoid (for bf16 it exceeds 2e-3 once |out| > ~1).
    Returns the max raw abs error.
    """
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape
    assert np.isfinite(g).all()
    rnd = np.abs(round_to_storage(ref, dtype) - ref)
    err = np.abs(g - ref)
    excess = err - rnd
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= tol, (f"max excess {excess.max():.3e} at {worst}: got {g[worst]} "
                                 f"ref {ref[worst]} (raw err {err.max():.3e})")
    return float(err.max())


def run_both(pa, w, params=None, keep_seqs=None, compare_cache=True, auto_share=True):
    """Replay w on the GPU (libpa) and on the oracle; compare traces, BM state, caches.

    auto_share: the engine's automatic choice of the shared-prefix decode for batches
    whose neighbouring sequences start on the same frame (off: always pa_decode's path).
    Returns (gpu outputs {op: tensor}, oracle result).
    """
    eng = pa.PagedKVEngine(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype,
                           free_order=w.free_order, max_seqs=max(64, len(w.final_lens)),
                           max_blocks_per_seq=max(1, max(-(-L // w.block_size) for L in w.final_lens.values())),
                           auto_share=auto_share)
    outs, trace = pa.run_workload_ops(eng, w, attend_params=params)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    ref = replay(w, keep_seqs=keep_seqs)
    # host block manager: every slot and copy pair, then the final state
    assert trace.pop("n_cached") == ref.n_cached
    for i, t in trace.items():
        assert t["slots"] == list(ref.trace[i]["slots"]), f"slots differ at op {i}"
        assert t["copies"] == [tuple(c) for c in ref.trace[i]["copies"]], f"copies differ at op {i}"
    assert eng.bm.free_list() == list(ref.bm.free_list)
    assert eng.bm.ref_counts() == ref.bm.refs
    for s, tab in ref.bm.tables.items():
        assert eng.bm.table(s) == tab
    if hasattr(ref.bm, "cached_frames"):
        assert eng.bm.cached_frames() == ref.bm.cached_frames()
    if compare_cache:
        if keep_seqs is None:
            assert np.array_equal(cache_bits(eng.k_cache), oracle_bits(ref.cache.k))
            assert np.array_equal(cache_bits(eng.v_cache), oracle_bits(ref.cache.v))
        else:
            for b in ref.cache.keep:
                assert np.array_equal(cache_bits(eng.k_cache[b]), oracle_bits(ref.cache.k[b])), b
                assert np.array_equal(cache_bits(eng.v_cache[b]), oracle_bits(ref.cache.v[b])), b
    return eng, outs, ref


def check_outputs(w, outs, ref, keep_seqs=None, tol: float = TOL) -> float:
    worst = 0.0
    for op_i, out in outs.items():
        r = ref.outputs[op_i]
        seqs = w.ops[op_i][1]
        idx = [j for j, s in enumerate(seqs) if keep_seqs is None or s in set(keep_seqs)]
        worst = max(worst, assert_attention_close(out[idx], r[idx], w.dtype, tol))
    return worst
