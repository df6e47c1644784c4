"""GPU parity of pa_prefill (causal attention for query chunks, tensor cores).

Gate, element-wise: |gpu - oracle| <= 2e-3 + half a unit in the last place of the
16-bit output (the rounding of the exact result to the output dtype, which no
kernel avoids).

Error model, checked as well (tighter).  The tensor cores take the softmax weights
in the cache's 16-bit type.  fp16 weights are rounded once: a result moves by at
most u * sum_j w_j |v_j|, u = 2^-11.  bf16 weights go as a high part plus the
remainder, two products into one fp32 accumulator: u = 2^-16.  Each weight is
formed once (the kernel fixes a tile's reference max before it forms any of the
tile's weights, so none is rescaled after rounding); ex2.approx and the fp32
accumulation add far less than 1e-4 here.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import prefill_weight_bound
from tests._gpu_common import run_both

pytestmark = pytest.mark.gpu

U_WEIGHTS = {"f16": 2.0 ** -11, "bf16": 2.0 ** -16}
MODEL_SLACK = 1e-4   # fp32 accumulation and ex2.approx, far above their size here
GATE = 2e-3

MANT = {"f16": 10, "bf16": 7}      # stored mantissa bits
MIN_EXP = {"f16": -14, "bf16": -126}


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit type at magnitude |x| (subnormal floor)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** MIN_EXP[dtype])))
    return 2.0 ** (e - MANT[dtype] - 1)


def check_prefill(w, outs, ref, keep=None, gate=GATE):
    """Gate and error model on every row, or on the rows of the sequences in ``keep``
    (positions in the prefill op's sequence list); returns the raw max abs error.
    The 2e-3 gate is stated for unit-scale values (N(0,1) or narrower): errors scale
    with |v|, so a test on wider values passes a gate scaled by their sigma."""
    (op,) = w.prefill_ops
    got_all = outs[op].double().cpu().numpy()
    tables, lens = ref.attend_meta[op]
    counts = list(w.ops[op][2])
    qs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    q = w.query(op)
    if keep is None:
        keep = range(len(counts))
    rows = np.concatenate([np.arange(qs[j], qs[j + 1]) for j in keep]).astype(np.int64)
    got, r = got_all[rows], ref.outputs[op][rows]
    assert np.isfinite(got).all()
    out_round = half_ulp(np.maximum(np.abs(got), np.abs(r)), w.dtype)
    err = np.abs(got - r)
    excess = err - out_round
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= gate, f"excess {excess.max():.3e} at {worst}: {got[worst]} vs {r[worst]}"
    sub_qs = np.concatenate([[0], np.cumsum([counts[j] for j in keep])]).astype(np.int64)
    bound = prefill_weight_bound(q[rows], ref.cache, [tables[j] for j in keep], [lens[j] for j in keep], sub_qs,
                                 w.scale)
    model = excess - U_WEIGHTS[w.dtype] * bound
    worst = np.unravel_index(np.argmax(model), model.shape)
    assert model.max() <= MODEL_SLACK, f"error model exceeded by {model.max():.3e} at {worst}"
    return float(err.max())


def test_small_prefill_batch(pa):
    w = workloads.prefill_batch(small=True)
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)


@pytest.mark.parametrize("prefix,chunk", [
    ([0], [1]), ([0], [127]), ([0], [128]), ([0], [129]), ([0], [300]),
    ([5], [1]), ([100], [1]), ([127], [1]), ([128], [1]), ([1000], [64]),
    ([0, 17, 256, 900], [513, 1, 128, 77]),
    # tile pairs: both tiles ending in the same key tile, odd tile counts, ragged tails
    ([5], [129]), ([0], [384]), ([60], [640]), ([200], [255]),
])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_chunks_and_prefixes(pa, prefix, chunk, dtype):
    w = workloads.chunked_prefill(prefix, chunk, H=2, D=128, B=16, dtype=dtype, seed=sum(prefix) + sum(chunk))
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
def test_block_sizes(pa, B):
    w = workloads.chunked_prefill([0, 300, 77], [200, 150, 260], H=3, D=128, B=B, dtype="f16", seed=B)
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)


def test_many_items_per_block(pa):
    """More work items than SMs: several items per persistent block, ring reuse."""
    rng = np.random.default_rng(5)
    pre = rng.integers(0, 700, size=10).tolist()
    ch = rng.integers(100, 400, size=10).tolist()
    w = workloads.chunked_prefill(pre, ch, H=8, D=128, B=16, dtype="bf16", seed=5)
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)
    # the work counter resets itself: a second launch gives the same bits
    (op,) = w.prefill_ops
    again = eng.prefill(w.ops[op][1], w.ops[op][2], w.query(op), w.scale)
    assert torch.equal(again, outs[op])
    assert pa.pa_get_device_status() == 0


def test_batch_larger_than_one_launch(pa):
    """5000 sequences of 1-3 query rows: more than one launch's shared memory holds (unit
    offsets and order per sequence), so pa_prefill runs consecutive ranges of sequences
    as separate launches, q and out whole."""
    rng = np.random.default_rng(41)
    pre = rng.integers(0, 40, size=5000).tolist()
    ch = rng.integers(1, 4, size=5000).tolist()
    w = workloads.chunked_prefill(pre, ch, H=2, D=128, B=16, dtype="f16", seed=41)
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)
    (op,) = w.prefill_ops
    n0 = pa.pa_launch_count()
    again = eng.prefill(w.ops[op][1], w.ops[op][2], w.query(op), w.scale)
    torch.cuda.synchronize()
    assert pa.pa_launch_count() - n0 >= 2
    assert torch.equal(again, outs[op])
    assert pa.pa_get_device_status() == 0


def test_prefill_one_query_matches_decode(pa):
    """A chunk of one query is a decode step: both kernels agree within tolerance."""
    L = [37, 300, 811, 1]
    w = workloads.chunked_prefill([x - 1 for x in L], [1] * len(L), H=4, D=128, B=16, dtype="f16", seed=9)
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref)
    (op,) = w.prefill_ops
    dec = eng.attend(w.ops[op][1], w.query(op), w.scale)
    assert (dec.float() - outs[op].float()).abs().max().item() < 2e-3


@pytest.mark.parametrize("sigma,dtype", [(3.0, "f16"), (4.0, "bf16")])
def test_wide_score_range(pa, sigma, dtype):
    """Scores with a spread of many log2 units: the reference max is raised from tile
    to tile (O and the row sums scaled in both halves alike), every weight still
    formed once.  Values are sigma times wider than the workloads', so the gate is
    too; the error model is absolute."""
    w = workloads.chunked_prefill([0, 700, 1500], [640, 300, 129], H=2, D=128, B=16, dtype=dtype, sigma=sigma,
                                  seed=int(sigma * 10))
    eng, outs, ref = run_both(pa, w)
    check_prefill(w, outs, ref, gate=GATE * sigma)


@pytest.mark.parametrize("qs_kind", ["past_end", "negative_start", "decreasing"])
def test_bad_query_ranges_flagged_and_skipped(pa, qs_kind):
    """A sequence whose query range leaves [0, T] (or runs backwards) is flagged with
    PA_DEV_BAD_LEN and its rows stay untouched; the other sequence is computed as in
    a clean launch."""
    w = workloads.chunked_prefill([40, 300], [200, 150], H=2, D=128, B=16, dtype="f16", seed=3)
    eng, outs, ref = run_both(pa, w)
    (op,) = w.prefill_ops
    seqs, counts = w.ops[op][1], w.ops[op][2]
    T = sum(counts)
    good = outs[op]
    dev = good.device
    assert pa.pa_get_device_status() == 0
    if qs_kind == "past_end":
        qs, bad_rows, ok_rows = [0, 200, T + 64], slice(200, T), slice(0, 200)
    elif qs_kind == "negative_start":
        qs, bad_rows, ok_rows = [-5, 200, T], slice(0, 200), slice(200, T)
    else:
        qs, bad_rows, ok_rows = [0, 200, 150], slice(200, T), slice(0, 200)
    tables, lens = eng.bm.block_tables(list(seqs), eng.max_blocks)
    q = pa.to_device_rows(w.query(op), w.dtype, dev)
    out = torch.full_like(good, 7.0)
    pa.pa_prefill(q, eng.k_cache, eng.v_cache, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                  torch.tensor(qs, dtype=torch.int32, device=dev), w.scale, out)
    assert pa.pa_get_device_status() & pa.PA_DEV_BAD_LEN
    assert torch.all(out[bad_rows] == 7.0)
    assert torch.equal(out[ok_rows], good[ok_rows])


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_full_size_prefill_batch(pa, dtype):
    """The timed chunked-prefill batch (16 sequences, prefix ~U[0, 3072], a 512-token
    chunk each, 32 heads) in both dtypes, in the launch configuration the bench times:
    the GPU computes every row; the oracle follows the sequences with the shortest and
    the longest context (whole chunks, all heads).  Prints the raw max error."""
    w = workloads.prefill_batch(dtype=dtype)
    (op,) = w.prefill_ops
    seqs = list(w.ops[op][1])
    by_len = sorted(seqs, key=lambda s: w.final_lens[s])
    keep = [by_len[0], by_len[-1]]
    eng, outs, ref = run_both(pa, w, keep_seqs=keep)
    err = check_prefill(w, outs, ref, keep=[seqs.index(s) for s in keep])
    print(f"{w.name}: raw max abs err {err:.3e} (gate {GATE})")
    assert pa.pa_get_device_status() == 0
