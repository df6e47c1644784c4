"""GPU parity of prefix caching: prompts admitted by token ids reuse the cached
blocks of an identical prefix (no K/V rows computed or written for them), and the
causal prefill of the remaining tokens runs over frames written by earlier requests.

Inputs: K/V rows are a function of the token prefix (as a model's would be), so
the oracle's prefill through reused frames is pinned to the definition on the CPU
(tests/test_oracle_prefix_cache.py); here the GPU is compared with that oracle,
with every slot, copy pair, table, reference count, cached-frame flag and cache
bit checked on the way.
"""

import numpy as np
import pytest
import torch

import workloads
from tests._gpu_common import run_both
from tests.test_gpu_prefill import GATE, MODEL_SLACK, U_WEIGHTS, half_ulp
from oracle import prefill_weight_bound

pytestmark = pytest.mark.gpu


def check_prefill_new(w, outs, ref):
    """The prefill gate (2e-3 beyond the output's own rounding) and the kernel's error
    model, as in the plain prefill tests."""
    for i, op in enumerate(w.ops):
        if op[0] != "prefill_new":
            continue
        tables, lens, counts = ref.attend_meta[i]
        got = outs[i].double().cpu().numpy()
        qs = w.position_queries(i)
        start = 0
        for j, s in enumerate(op[1]):
            g = got[start:start + counts[j]]
            start += counts[j]
            r = ref.outputs[i][j]
            q = qs[j][lens[j] - counts[j]:lens[j]]
            bound = prefill_weight_bound(q, ref.cache, [tables[j]], [lens[j]], [0, counts[j]], w.scale)
            assert np.isfinite(g).all()
            excess = np.abs(g - r) - half_ulp(np.maximum(np.abs(g), np.abs(r)), w.dtype)
            assert excess.max() <= GATE, (i, s, excess.max())
            model = excess - U_WEIGHTS[w.dtype] * bound
            assert model.max() <= MODEL_SLACK, (i, s, model.max())
        assert start == got.shape[0]


@pytest.mark.parametrize("turns,free_between,B,dtype", [
    (1, False, 16, "f16"), (2, False, 16, "f16"), (3, True, 16, "bf16"), (2, False, 32, "f16"), (2, True, 8, "bf16"),
])
def test_shared_prefix_turns(pa, turns, free_between, B, dtype):
    w = workloads.shared_prefix(4, 300, [130, 17, 256, 1], H=2, B=B, dtype=dtype, turns=turns, reply_len=40,
                                free_between=free_between, seed=40 + turns + B)
    eng, outs, ref = run_both(pa, w)
    assert sum(ref.n_cached.values()) > 0
    check_prefill_new(w, outs, ref)


def test_reuse_writes_only_uncached_rows(pa):
    """A second identical request computes one token: its admission writes one row."""
    w = workloads.shared_prefix(1, 64, [0], H=2, B=16, seed=3)
    eng, outs, ref = run_both(pa, w)
    toks = list(w.ops[0][2])
    before = eng.k_cache.clone()
    n_cached, slots = eng.add_seq_cached(99, toks)
    assert n_cached == 48 and len(slots) == 16        # the last block holds the last token: recomputed
    k, v = w.prefix_rows(toks)
    eng.write_rows(slots, k[n_cached:], v[n_cached:])
    torch.cuda.synchronize()
    # the shared frames were not touched; the new frame holds the same bits as the first request's
    t0, t1 = eng.bm.table(0), eng.bm.table(99)
    assert t1[:3] == t0[:3] and t1[3] != t0[3]
    assert torch.equal(eng.k_cache[t0[:3]], before[t0[:3]])
    assert torch.equal(eng.k_cache[t1[3]], eng.k_cache[t0[3]])
