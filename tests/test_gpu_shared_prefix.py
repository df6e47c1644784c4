"""GPU parity of the shared-prefix decode (pa_decode_ex with share_prefix) against the
oracle.

The result must be pa_decode's: softmax attention of each sequence over its own
tokens, within 2e-3 of the fp64 oracle.  Cases cover the chunking rules (runs longer
than one chunk, shared lengths that vary inside a run, identical tables, contexts that
are entirely shared, empty and invalid lengths that end a run), every built launch
shape, block sizes 8..64, forced small, whole and automatic parts, poisoned frames in
a shared prefix, and the fork workloads replayed end to end through the engine.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import OracleKVCache, paged_decode
from tests._gpu_common import assert_attention_close, check_outputs, run_both

pytestmark = pytest.mark.gpu


def _tree(specs, B, seed):
    """Block tables from (parent, kept_frames, length) specs: a sequence copies the first
    kept_frames entries of its parent's table (parent None: none) and takes fresh frames
    for the rest.  Frame ids come from a shuffled pool."""
    rng = np.random.default_rng(seed)
    need = sum(-(-L // B) for _, _, L in specs) + 4
    pool = list(rng.permutation(need))
    tables = []
    for parent, kept, L in specs:
        nblk = -(-L // B)
        t = list(tables[parent][:kept]) if parent is not None else []
        while len(t) < nblk:
            t.append(int(pool.pop()))
        tables.append(t[:max(nblk, len(t))])
    return tables, need


def _run(pa, specs, *, B, H=4, dtype="f16", params=None, seed=0, lens_override=None, table_edit=None, sigma=1.0,
         tol=2e-3):
    tables, nb = _tree(specs, B, seed)
    lens = [L for _, _, L in specs]
    if lens_override:
        for i, L in lens_override.items():
            lens[i] = L
    if table_edit:
        table_edit(tables)
    S, D = len(specs), 128
    mb = max(1, max(len(t) for t in tables))
    kc = workloads.random_storage(seed + 1, (nb, B, H, D), dtype, sigma)
    vc = workloads.random_storage(seed + 2, (nb, B, H, D), dtype, sigma)
    q = workloads.random_storage(seed + 3, (S, H, D), dtype, sigma)
    dev = torch.device("cuda")
    td = torch.full((S, mb), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        td[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
    kd = pa.to_device_rows(kc.reshape(nb * B, H, D), dtype, dev).view(nb, B, H, D)
    vd = pa.to_device_rows(vc.reshape(nb * B, H, D), dtype, dev).view(nb, B, H, D)
    qd = pa.to_device_rows(q, dtype, dev)
    out = torch.full_like(qd, 7.0)
    scale = float(np.float32(1.0 / np.sqrt(D)))
    p = {"share_prefix": B}
    p.update(params or {})
    pa.pa_decode_ex(qd, kd, vd, td.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev), scale, out, p)
    torch.cuda.synchronize()
    cache = OracleKVCache(nb, B, H, D, dtype)
    cache.k[...] = kc
    cache.v[...] = vc
    ok = [s for s in range(S) if 0 <= lens[s] <= mb * B and all(0 <= f < nb for f in tables[s][:-(-lens[s] // B)])]
    ref = paged_decode(q[ok], cache, [tables[s] for s in ok], [lens[s] for s in ok], scale)
    assert_attention_close(out[ok], ref, dtype, tol)
    return out, lens, tables


def _siblings(n, prompt, B, tails, seed=0):
    """n forks of one prompt (the last frame copied on divergence when it is partial),
    then private tails of the given lengths."""
    rng = np.random.default_rng(seed)
    kept = prompt // B  # full frames shared; a partial last frame is copied by a writer
    specs = [(None, 0, prompt + tails[0])]
    for i in range(1, n):
        specs.append((0, kept, prompt + tails[i % len(tails)] + int(rng.integers(0, 3))))
    return specs


SHAPES = [(4, 1), (2, 1), (1, 1)]


@pytest.mark.parametrize("hg,wph", SHAPES)
@pytest.mark.parametrize("B", [8, 16, 32, 64])
@pytest.mark.parametrize("part", [0, -1, 2])
def test_runs_chunks_and_shapes(pa, hg, wph, B, part):
    """19 siblings (chunks of 16 and 3), then unrelated sequences and another family."""
    specs = _siblings(19, 37 * B // 2 + 3, B, [0, 5, 17, 40, 1, 64])
    base = len(specs)
    specs += [(None, 0, 100), (None, 0, 7 * B)]
    specs += [(base + 1, 5, 7 * B + 9), (base + 1, 7, 7 * B), (base + 1, 3, 3 * B + 2)]
    params = {"heads_per_cta": hg, "warps_per_head": wph, "partition_tokens": part * B if part > 0 else part}
    for dtype in ("f16", "bf16"):
        _run(pa, specs, B=B, H=4, dtype=dtype, params=params, seed=B + hg)
    assert pa.pa_get_device_status() == 0


def test_shared_length_varies_inside_a_run(pa):
    B = 16
    specs = [(None, 0, 700), (0, 40, 690), (1, 20, 400), (0, 38, 650), (3, 38, 660), (4, 10, 170)]
    for part in (0, -1, 3 * B):
        _run(pa, specs, B=B, params={"partition_tokens": part}, seed=3)


@pytest.mark.parametrize("L", [333, 320, 16, 17, 1])
def test_identical_tables_whole_context_shared(pa, L):
    """Forks that have not appended yet: identical tables and lengths.  When L is a
    frame multiple the whole context is shared (no private part)."""
    B = 16
    specs = [(None, 0, L)] + [(0, 10 ** 6, L)] * 5
    for part in (0, -1, B):
        _run(pa, specs, B=B, params={"partition_tokens": part}, seed=L)


def test_empty_and_invalid_lengths_end_runs(pa):
    B = 16
    specs = [(None, 0, 300), (0, 18, 300), (0, 18, 310), (0, 18, 305), (0, 18, 320), (0, 18, 299)]
    out, lens, _ = _run(pa, specs, B=B, lens_override={2: 0}, seed=4)
    assert torch.all(out[2] == 0)
    assert pa.pa_get_device_status() == 0
    out, lens, _ = _run(pa, specs, B=B, lens_override={3: 10 ** 6}, seed=5)
    assert torch.all(out[3] == 0)
    assert pa.pa_get_device_status() == pa.PA_DEV_BAD_LEN


def test_bad_frame_in_shared_prefix_zeroes_every_member(pa):
    B = 16
    specs = [(None, 0, 400), (0, 25, 410), (0, 25, 420), (0, 25, 405), (None, 0, 200)]

    def poison(tables):
        for s in range(4):
            tables[s][3] = 10 ** 6
    for part in (0, -1, 2 * B):
        out, _, _ = _run(pa, specs, B=B, table_edit=poison, params={"partition_tokens": part}, seed=6)
        assert torch.all(out[:4] == 0)
        assert pa.pa_get_device_status() & pa.PA_DEV_BAD_BLOCK


def test_threshold_and_no_sharing(pa):
    """Below the threshold nothing is grouped; unrelated sequences only: same results."""
    B = 16
    specs = _siblings(6, 200, B, [3, 9])
    for thr in (1, B, 256, 10 ** 6):
        _run(pa, specs, B=B, params={"share_prefix": thr}, seed=7)
    _run(pa, [(None, 0, L) for L in (1, 50, 300, 17, 0, 900)], B=B, seed=8)


def test_repeated_launches_identical(pa):
    B = 16
    specs = _siblings(8, 500, B, [0, 30, 70, 200])
    out0, _, _ = _run(pa, specs, B=B, seed=9)
    for _ in range(3):
        out1, _, _ = _run(pa, specs, B=B, seed=9)
        assert torch.equal(out0, out1)


def test_options_validated(pa):
    B, H, D = 16, 4, 128
    kc = torch.zeros(4, B, H, D, device="cuda", dtype=torch.float16)
    q = torch.zeros(2, H, D, device="cuda", dtype=torch.float16)
    t = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    lens = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(pa.PAError):
        pa.pa_decode_ex(q, kc, kc, t, lens, 1.0, out, {"share_prefix": -1})
    with pytest.raises(pa.PAError):  # launch shape not built for the shared-prefix kernel
        pa.pa_decode_ex(q, kc, kc, t, lens, 1.0, out, {"share_prefix": 1, "heads_per_cta": 1, "warps_per_head": 2})
    with pytest.raises(ValueError):
        pa.pa_decode_ex(q, kc, kc, t, lens, 1.0, out, {"share_prefixes": 1})
    # shapes the shared-prefix kernel does not take run the plain decode
    k64 = torch.zeros(4, B, H, 64, device="cuda", dtype=torch.float16)
    q64 = torch.zeros(2, H, 64, device="cuda", dtype=torch.float16)
    pa.pa_decode_ex(q64, k64, k64, t, lens, 1.0, torch.zeros_like(q64), {"share_prefix": 1})
    assert pa.pa_get_device_status() == 0


# ---- fork workloads end to end through the engine --------------------------------------------
@pytest.mark.parametrize("cfg", [3, 2, 4])
def test_config_workloads(pa, cfg):
    w = workloads.build(cfg, small=True)
    eng, outs, ref = run_both(pa, w, params={"share_prefix": w.block_size})
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("width,B,dtype", [(4, 16, "f16"), (8, 8, "bf16"), (3, 32, "f16")])
def test_beam_search(pa, width, B, dtype):
    w = workloads.beam_search(3, 300, width, 24, H=4, B=B, dtype=dtype, seed=50 + width)
    eng, outs, ref = run_both(pa, w, params={"share_prefix": B})
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("batch,B,dtype", [(4, 16, "f16"), (8, 8, "bf16")])
def test_mcts(pa, batch, B, dtype):
    w = workloads.mcts_tree(2, 200, 12, batch=batch, rollout_max=40, max_nodes=30, H=4, B=B, dtype=dtype,
                            seed=60 + batch)
    eng, outs, ref = run_both(pa, w, params={"share_prefix": B})
    check_outputs(w, outs, ref)


def test_many_sequences(pa):
    """2000 sequences: runs of 1..16 siblings of short prompts, the plan's scans over many
    32-sequence rounds, thousands of parts."""
    B = 16
    rng = np.random.default_rng(21)
    specs = []
    while len(specs) < 2000:
        n = int(rng.integers(1, 17))
        root = len(specs)
        base = int(rng.integers(20, 200))
        specs.append((None, 0, base))
        for _ in range(n - 1):
            specs.append((root, base // B, base + int(rng.integers(0, 40))))
    specs = specs[:2000]
    _run(pa, specs, B=B, H=2, params={"share_prefix": B}, seed=22)
    _run(pa, specs, B=B, H=2, params={"share_prefix": B, "partition_tokens": B}, seed=23)
    assert pa.pa_get_device_status() == 0


def test_long_shared_prefix(pa):
    """Four siblings over a 65536-token prompt: many shared parts per chunk."""
    B = 64
    specs = [(None, 0, 65536 + 5)] + [(0, 65536 // B, 65536 + t) for t in (0, 100, 3)]
    for part in (0, 1024):
        _run(pa, specs, B=B, H=2, params={"share_prefix": 1, "partition_tokens": part}, seed=24)
    assert pa.pa_get_device_status() == 0


@pytest.mark.parametrize("sigma", [3.0, 4.0])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_wide_value_range(pa, sigma, dtype):
    """Queries, keys and values of spread sigma: scores of spread sigma^2, so a row's
    reference max moves often and its weights span many binades.  The 2e-3 gate holds
    for unit-scale values; the fp32 score error grows with |q||k|, so the gate scales with
    sigma here."""
    B = 16
    specs = _siblings(9, 40 * B + 5, B, [0, 3, 70, 200], seed=9)
    for part in (0, 2 * B):
        _run(pa, specs, B=B, dtype=dtype, params={"partition_tokens": part}, seed=31, sigma=sigma,
             tol=2e-3 * sigma)
    assert pa.pa_get_device_status() == 0
