"""Full-size GPU parity on the five workloads, in the launch configuration the bench
times (automatic launch parameters).

Decode batch (64 x U[512,2048], f16), the fixed 64 x 2048 batch, long context
(4 x 16384, bf16, split + merge), parallel sampling with copy-on-write
(16 prompts x 4 branches) and the serving mix (256 sequences, log-uniform lengths
up to 8192, 40 heads, bf16, one appended token each before attention): every slot,
copy pair, block-manager state, the whole cache bit for bit, and every attention
output against the oracle.
"""

import functools

import pytest

import workloads
from tests._gpu_common import check_outputs, run_both

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("cfg", [1, "1x", 2, 3])
def test_full_workload(pa, cfg):
    w = workloads.build(cfg)
    eng, outs, ref = run_both(pa, w)
    err = check_outputs(w, outs, ref)
    print(f"{w.name}: max abs err {err:.2e}")


def test_serving_mix_full(pa):
    """All 256 sequences.  The ~8 GB of K/V rows are drawn once by the workload
    generator and handed to both sides (the engine's replay and the oracle's), which
    stay independent otherwise."""
    w = workloads.build(4)
    w.rows = functools.lru_cache(maxsize=None)(w.rows)
    eng, outs, ref = run_both(pa, w)
    err = check_outputs(w, outs, ref)
    print(f"{w.name}: all {len(w.final_lens)} seqs, max abs err {err:.2e}")
