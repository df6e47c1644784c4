"""Full-size GPU parity on the five workloads, in the launch configuration the bench
times (automatic launch parameters).

Decode batch (64 x U[512,2048], f16), the fixed 64 x 2048 batch, long context
(4 x 16384, bf16, split + merge) and parallel sampling with copy-on-write
(16 prompts x 4 branches): every slot, copy pair, block-manager state, the whole
cache bit for bit, and every attention output against the oracle.  Serving mix
(256 sequences, log-uniform lengths up to 8192, 40 heads, bf16): the oracle
follows a sample of sequences (shortest, longest and random ones); their frames
are compared bit for bit and their outputs within tolerance.
"""

import numpy as np
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


def test_serving_mix_sampled(pa):
    w = workloads.build(4)
    lens = w.final_lens
    order = sorted(lens, key=lambda s: lens[s])
    rng = np.random.default_rng(4)
    keep = sorted(set(order[:3] + order[-3:] + rng.choice(len(lens), 10, replace=False).tolist()))
    eng, outs, ref = run_both(pa, w, keep_seqs=keep)
    err = check_outputs(w, outs, ref, keep_seqs=keep)
    print(f"{w.name}: sampled {len(keep)} seqs, max abs err {err:.2e}")
