"""GPU parity of the CUDA path against the oracle (small and edge-case workloads).

Everything runs through libpa's C ABI: host block manager, pa_copy_blocks,
pa_cache_append, pa_decode (+ merge).  Block state, slot mappings, copy pairs and
the whole cache must be bit-exact; attention outputs within 2e-3 of the fp64
oracle (plus the unavoidable rounding of the exact result to the output dtype).
"""

import math

import numpy as np
import pytest
import torch

import workloads
from tests._gpu_common import TOL, assert_attention_close, check_outputs, run_both

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [0, 1, "1x", 2, 3, 4])
def test_small_workloads(pa, cfg):
    w = workloads.build(cfg, small=True) if cfg != 0 else workloads.build(0)
    eng, outs, ref = run_both(pa, w)
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
@pytest.mark.parametrize("mode", ["never", "forced", "auto"])
def test_split_modes_agree_with_oracle(pa, cfg, mode):
    w = workloads.build(cfg, small=True)
    params = {"never": {"partition_tokens": -1}, "forced": {"partition_tokens": 2 * w.block_size},
              "auto": None}[mode]
    eng, outs, ref = run_both(pa, w, params=params)
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("hg,wph", [(1, 1), (1, 2), (1, 4), (1, 8), (2, 1), (2, 2), (2, 4), (4, 1), (4, 2)])
@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("B,dtype", [(16, "f16"), (32, "bf16")])
def test_launch_shapes(pa, hg, wph, stages, B, dtype):
    """Every built (heads per block, warps per head) pair; B = 16 * warps per head takes
    the unrolled full-frame path, the rest (and every partly filled frame) the generic one."""
    w = workloads.custom([1, 15, 16, 17, 33, 200, 333, 700], H=8, D=128, B=B, dtype=dtype, seed=11)
    params = {"heads_per_cta": hg, "warps_per_head": wph, "stages": stages, "partition_tokens": 4 * B}
    eng, outs, ref = run_both(pa, w, params=params)
    check_outputs(w, outs, ref)


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_generic_path_on_fast_shapes(pa, cfg):
    w = workloads.build(cfg, small=True)
    eng, outs, ref = run_both(pa, w, params={"generic_only": 1})
    check_outputs(w, outs, ref)


def test_repeated_launches_identical(pa):
    """The work counter resets itself: back-to-back launches, on one stream and on two
    streams, give the same bits."""
    w = workloads.custom([300, 1000, 17, 4000, 2048], H=8, D=128, B=16, dtype="f16", seed=21)
    eng, outs, ref = run_both(pa, w)
    (op,) = [i for i, o in enumerate(w.ops) if o[0] == "attend"]
    q = pa.to_device_rows(w.query(op), w.dtype, eng.device)
    first = outs[op].clone()
    for _ in range(5):
        again = eng.attend(w.ops[op][1], q, w.scale)
        assert torch.equal(again, first)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        again = eng.attend(w.ops[op][1], q, w.scale)
    side.synchronize()
    assert torch.equal(again, first)
    for items in (1, 2, 16):
        o = eng.attend(w.ops[op][1], q, w.scale, params={"items_per_cta": items})
        assert_attention_close(o, ref.outputs[op], w.dtype)
    assert pa.pa_get_device_status() == 0


EDGE = [
    # (lengths, H, D, B, dtype)
    ([0, 1, 2, 9, 10, 11, 19, 20, 21], 2, 64, 10, "f32"),
    ([1, 15, 16, 17, 31, 32, 33], 3, 128, 16, "f16"),
    ([1, 31, 32, 33, 255, 256, 257, 512, 513], 4, 128, 32, "bf16"),
    ([5, 64, 300], 2, 256, 16, "bf16"),
    ([5, 64, 300], 1, 256, 8, "f16"),
    ([7, 100, 129], 4, 64, 16, "f16"),
    ([3, 40, 77], 5, 128, 16, "f32"),
    ([1, 2, 3, 4], 40, 128, 16, "bf16"),
    ([600, 1], 2, 128, 1, "f16"),            # one token per frame
    ([256 * 3 + 1], 2, 64, 256, "f16"),      # largest supported frame
]


@pytest.mark.parametrize("lengths,H,D,B,dtype", EDGE)
@pytest.mark.parametrize("part", [0, -1, 1])
def test_edge_cases(pa, lengths, H, D, B, dtype, part):
    w = workloads.custom(lengths, H=H, D=D, B=B, dtype=dtype, seed=sum(lengths) + H)
    params = {"partition_tokens": B if part == 1 else part}
    eng, outs, ref = run_both(pa, w, params=params)
    check_outputs(w, outs, ref)


def test_physical_permutation_gives_identical_bits(pa):
    """Relabelling physical frames changes no output bit (order of arithmetic fixed)."""
    L = [37, 300, 811, 1]
    results = []
    for seed in range(3):
        base = workloads.custom(L, H=4, D=128, B=16, dtype="f16", seed=5)
        order = np.random.default_rng(seed).permutation(base.num_blocks).astype(np.int32)
        w = workloads.custom(L, H=4, D=128, B=16, dtype="f16", seed=5, free_order=order)
        eng, outs, ref = run_both(pa, w, params={"partition_tokens": 128})
        (o,) = outs.values()
        results.append(o.view(torch.int16).cpu().numpy())
    for r in results[1:]:
        assert np.array_equal(r, results[0])


def test_identity_table_matches_torch_attention(pa):
    """Contiguous frames (identity table) == dense attention in plain PyTorch fp32."""
    torch.manual_seed(0)
    B, H, D, L = 16, 4, 128, 1000
    nb = -(-L // B)
    k = torch.randn(nb * B, H, D, device="cuda").half()
    v = torch.randn(nb * B, H, D, device="cuda").half()
    q = torch.randn(1, H, D, device="cuda").half()
    kc, vc = k.view(nb, B, H, D).contiguous(), v.view(nb, B, H, D).contiguous()
    table = torch.arange(nb, dtype=torch.int32, device="cuda")[None]
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    for part in (-1, 0, 64):
        out = torch.empty_like(q)
        pa.pa_decode(q, kc, vc, table, lens, scale, out, params={"partition_tokens": part})
        a = torch.einsum("hd,lhd->hl", q[0].float(), k[:L].float()) * scale
        ref = torch.einsum("hl,lhd->hd", torch.softmax(a, dim=-1), v[:L].float())
        assert (out[0].float() - ref).abs().max().item() < TOL


def test_bad_indices_set_status_and_zero_rows(pa):
    """Poisoned table entries / lengths / slots / copy ids: checked, skipped, reported."""
    B, H, D = 16, 2, 64
    nb = 8
    kc = torch.randn(nb, B, H, D, device="cuda").half()
    vc = torch.randn(nb, B, H, D, device="cuda").half()
    q = torch.randn(3, H, D, device="cuda").half()
    table = torch.tensor([[0, 1, 2], [3, nb + 5, 4], [5, 6, -3]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([40, 40, 48], dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    assert pa.pa_get_device_status() == 0
    pa.pa_decode(q, kc, vc, table, lens, 0.125, out, params={"partition_tokens": -1})
    st = pa.pa_get_device_status()
    assert st & pa.PA_DEV_BAD_BLOCK
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    assert torch.isfinite(out[0]).all() and not torch.all(out[0] == 0)
    # forced split path: the merge also zeroes poisoned rows
    out.fill_(7.0)
    pa.pa_decode(q, kc, vc, table, lens, 0.125, out, params={"partition_tokens": 16})
    assert pa.pa_get_device_status() & pa.PA_DEV_BAD_BLOCK
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    # context longer than the table allows
    lens_bad = torch.tensor([40, 1000, -2], dtype=torch.int32, device="cuda")
    out.fill_(7.0)
    pa.pa_decode(q, kc, vc, table, lens_bad, 0.125, out)
    assert pa.pa_get_device_status() & pa.PA_DEV_BAD_LEN
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    # out-of-range slot: skipped, reported; padding slot -1 silently skipped
    before = kc.clone()
    rows = torch.randn(3, H, D, device="cuda").half()
    slots = torch.tensor([nb * B, -1, 5], dtype=torch.int32, device="cuda")
    pa.pa_cache_append(rows, rows, slots, kc, vc)
    assert pa.pa_get_device_status() == pa.PA_DEV_BAD_SLOT
    expect = before.view(-1, H, D).clone()
    expect[5] = rows[2]
    assert torch.equal(kc.view(-1, H, D), expect)
    # bad copy pair
    pairs = torch.tensor([[0, nb], [1, 2]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, pairs)
    assert pa.pa_get_device_status() == pa.PA_DEV_BAD_COPY
    assert torch.equal(kc[2], kc[1])
    assert pa.pa_get_device_status() == 0


def test_host_validation_errors(pa):
    B, H, D = 16, 2, 64
    kc = torch.zeros(4, B, H, D, device="cuda", dtype=torch.float16)
    q = torch.zeros(1, H, D, device="cuda", dtype=torch.float16)
    t = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(pa.PAError):   # dtype mismatch
        pa.pa_decode(q.float(), kc, kc, t, lens, 1.0, out.float())
    with pytest.raises(pa.PAError):   # head_dim not built
        k2 = torch.zeros(4, B, H, 48, device="cuda", dtype=torch.float16)
        pa.pa_decode(torch.zeros(1, H, 48, device="cuda", dtype=torch.float16), k2, k2, t, lens, 1.0,
                     torch.zeros(1, H, 48, device="cuda", dtype=torch.float16))
    with pytest.raises(pa.PAError):   # non-contiguous cache
        kt = torch.zeros(4, H, B, D, device="cuda", dtype=torch.float16).transpose(1, 2)
        pa.pa_decode(q, kt, kt, t, lens, 1.0, out)
    with pytest.raises(pa.PAError):   # shape mismatch of lengths
        pa.pa_decode(q, kc, kc, t, torch.zeros(2, dtype=torch.int32, device="cuda"), 1.0, out)
    with pytest.raises(pa.PAError):   # bad option
        pa.pa_decode(q, kc, kc, t, lens, 1.0, out, params={"heads_per_cta": 3})
    # an empty batch is a no-op
    pa.pa_decode(q[:0], kc, kc, t[:0], lens[:0], 1.0, out[:0])
    assert pa.pa_get_device_status() == 0


def test_many_sequences_prefix_scan(pa):
    """More sequences than one warp's scan chunk; lengths 0..B*3 mixed."""
    rng = np.random.default_rng(3)
    L = rng.integers(0, 49, size=333).tolist()
    w = workloads.custom(L, H=2, D=64, B=16, dtype="f16", seed=3)
    eng, outs, ref = run_both(pa, w, params={"partition_tokens": 16})
    check_outputs(w, outs, ref)


def test_batch_larger_than_one_launch(pa):
    """24,000 sequences: more than one launch holds (every thread block keeps three
    int32 per sequence in shared memory), so pa_decode runs consecutive ranges of
    sequences as separate launches; every output against the oracle."""
    rng = np.random.default_rng(31)
    L = rng.integers(1, 13, size=24000).tolist()
    w = workloads.custom(L, H=2, D=64, B=8, dtype="f16", seed=31)
    eng, outs, ref = run_both(pa, w)
    check_outputs(w, outs, ref)
    (op,) = [i for i, o in enumerate(w.ops) if o[0] == "attend"]
    q = pa.to_device_rows(w.query(op), w.dtype, eng.device)
    n0 = pa.pa_launch_count()
    again = eng.attend(w.ops[op][1], q, w.scale)
    torch.cuda.synchronize()
    assert pa.pa_launch_count() - n0 >= 2
    assert torch.equal(again, outs[op])
    # the fixed-scratch entry point launches once or refuses
    tables, lens = eng.bm.block_tables(w.ops[op][1], eng.max_blocks)
    tt, ll = torch.from_numpy(tables).to(eng.device), torch.from_numpy(lens).to(eng.device)
    with pytest.raises(pa.PAError):
        pa.pa_decode_static(q, eng.k_cache, eng.v_cache, tt, ll, w.scale, torch.empty_like(q))
    assert pa.pa_get_device_status() == 0


@pytest.mark.parametrize("sigma", [3.0, 4.0])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_wide_value_range(pa, sigma, dtype):
    """Queries, keys and values of spread sigma (scores of spread sigma^2): the running
    max moves often and weights span many binades, whole and split into partitions.  The
    2e-3 gate holds for unit-scale values; the fp32 score error grows with |q||k|, so the
    gate scales with sigma here."""
    w = workloads.custom([1, 17, 300, 1000, 2500], H=4, D=128, B=16, dtype=dtype, sigma=sigma, seed=int(sigma) + 40)
    for part in (0, -1, 64):
        eng, outs, ref = run_both(pa, w, params={"partition_tokens": part})
        check_outputs(w, outs, ref, tol=2e-3 * sigma)
    assert pa.pa_get_device_status() == 0
