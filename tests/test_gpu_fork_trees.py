"""GPU parity on fork-tree workloads: beam search and MCTS over forked sequences.

Every decode attention reads prompts shared by many branches; every step moves
writers of shared tails onto private copies (pa_copy_blocks) before appending.  Each
workload runs twice: through pa_decode, and through the engine's automatic choice of the
shared-prefix decode (the batches' neighbouring beams start on the same frames).
All slots, copy pairs, tables, reference counts and cache bits are compared with
the oracle after the replay, and every attention output element-wise.
"""

import pytest

import workloads
from tests._gpu_common import check_outputs, run_both

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("auto_share", [False, True])
@pytest.mark.parametrize("width,B,dtype", [(4, 16, "f16"), (8, 8, "bf16"), (3, 32, "f16")])
def test_beam_search(pa, width, B, dtype, auto_share):
    w = workloads.beam_search(3, 300, width, 24, H=4, B=B, dtype=dtype, seed=50 + width)
    eng, outs, ref = run_both(pa, w, auto_share=auto_share)
    assert sum(len(t["copies"]) for t in ref.trace.values()) > 0
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("auto_share", [False, True])
@pytest.mark.parametrize("batch,B,dtype", [(4, 16, "f16"), (8, 8, "bf16")])
def test_mcts(pa, batch, B, dtype, auto_share):
    w = workloads.mcts_tree(2, 200, 12, batch=batch, rollout_max=40, max_nodes=30, H=4, B=B, dtype=dtype,
                            seed=60 + batch)
    eng, outs, ref = run_both(pa, w, auto_share=auto_share)
    check_outputs(w, outs, ref)
