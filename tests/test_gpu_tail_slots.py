"""Cache slots that hold no token of a sequence may contain anything (GPU).

A decode reads whole frames, so the slots of a sequence's last frame past its length,
and frames no table names, are read but must not change the result: their keys are
masked and their values must not enter the weighted sum (0 times a non-finite value
is not 0).  Here every such slot holds NaN, the written slots random finite values,
and each decode path must match the oracle, which reads only the sequence's own tokens
(pa_decode whole, split into partitions with the merge, automatic; the shared-prefix
decode; pa_decode_static; pa_decode_split on the same caches permuted into the pages'
split layout).  pa_prefill's value product runs on the tensor cores, where a zero
weight times a non-finite value would not vanish: its contract asks those slots to hold
finite values, and its test fills them with the largest finite values instead.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import OracleKVCache, paged_decode, paged_prefill, split_layout
from tests._gpu_common import assert_attention_close
from tests.test_gpu_prefill import GATE, MODEL_SLACK, U_WEIGHTS, half_ulp
from oracle import prefill_weight_bound

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}


MAX_BITS = {"f16": 0x7BFF, "bf16": 0x7F7F}  # largest finite value of the type


def _case(dtype, seed, filler=None):
    B, H, D = 16, 4, 128
    L = [1, 15, 17, 300, 300, 777, 0, 33, 64, 65]
    need = sum(-(-x // B) for x in L) + 4
    order = np.random.default_rng(seed).permutation(need)
    tables, pos = [], 0
    mb = max(-(-x // B) for x in L)
    for x in L:
        n = -(-x // B)
        tables.append([int(f) for f in order[pos:pos + n]] + [-1] * (mb - n))
        pos += n
    # sequences 3 and 4 share their first 16 frames (a fork), so the shared-prefix path
    # has a run to read once
    tables[4][:16] = tables[3][:16]
    bits = {}
    for kind, sd in (("k", 1), ("v", 2)):
        full = workloads.random_storage(seed + sd, (need, B, H, D), dtype).view(np.uint16).copy()
        live = np.zeros((need, B), bool)
        for t, x in zip(tables, L):
            for j in range(-(-x // B)):
                live[t[j], : min(B, x - j * B)] = True
        full[~live] = NAN_BITS[dtype] if filler is None else filler[dtype]
        bits[kind] = full
    q = workloads.random_storage(seed + 3, (len(L), H, D), dtype)
    return B, H, D, L, tables, bits, q


def _oracle(dtype, B, H, D, L, tables, bits, q, scale):
    need = bits["k"].shape[0]
    c = OracleKVCache(need, B, H, D, dtype)
    c.k = bits["k"].view(np.float16) if dtype == "f16" else bits["k"]
    c.v = bits["v"].view(np.float16) if dtype == "f16" else bits["v"]
    return paged_decode(q, c, [t for t in tables], L, scale)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_unwritten_slots_never_reach_the_output(pa, dtype):
    B, H, D, L, tables, bits, q = _case(dtype, seed=31)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    ref = _oracle(dtype, B, H, D, L, tables, bits, q, scale)
    dev = torch.device("cuda")
    kc = torch.from_numpy(bits["k"].view(np.int16)).to(dev).view(TD[dtype])
    vc = torch.from_numpy(bits["v"].view(np.int16)).to(dev).view(TD[dtype])
    qd = torch.from_numpy(q.view(np.int16)).to(dev).view(TD[dtype])
    td = torch.tensor(np.array(tables, np.int32), device=dev)
    ld = torch.tensor(L, dtype=torch.int32, device=dev)
    for params in ({}, {"partition_tokens": -1}, {"partition_tokens": 32}, {"share_prefix": 16}, "static"):
        out = torch.empty_like(qd)
        if params == "static":
            pa.pa_decode_static(qd, kc, vc, td, ld, scale, out)
        else:
            pa.pa_decode_ex(qd, kc, vc, td, ld, scale, out, params)
        torch.cuda.synchronize()
        assert pa.pa_get_device_status() == 0, params
        assert_attention_close(out, ref, dtype)
    # the pages' split layout, same values (NaN where nothing was written)
    ks, vs = split_layout(bits["k"], bits["v"], 2)
    ksd = torch.from_numpy(ks.view(np.int16)).to(dev).view(TD[dtype]).reshape(ks.shape[0], H, D // 8, B * 8)
    vsd = torch.from_numpy(vs.view(np.int16)).to(dev).view(TD[dtype])
    out = torch.empty_like(qd)
    pa.pa_decode_split(qd, ksd, vsd, td, ld, scale, out)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    assert_attention_close(out, ref, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_ignores_unwritten_slots(pa, dtype):
    B, H, D, L, tables, bits, q = _case(dtype, seed=41, filler=MAX_BITS)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    # the last n_s positions of every non-empty sequence are the chunk's queries
    counts = [min(x, c) for x, c in zip(L, [1, 15, 17, 130, 129, 300, 0, 33, 64, 65])]
    qs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    qrows = workloads.random_storage(51, (int(qs[-1]), H, D), dtype)
    need = bits["k"].shape[0]
    c = OracleKVCache(need, B, H, D, dtype)
    c.k = bits["k"].view(np.float16) if dtype == "f16" else bits["k"]
    c.v = bits["v"].view(np.float16) if dtype == "f16" else bits["v"]
    ref = paged_prefill(qrows, c, tables, L, qs, scale)
    dev = torch.device("cuda")
    kc = torch.from_numpy(bits["k"].view(np.int16)).to(dev).view(TD[dtype])
    vc = torch.from_numpy(bits["v"].view(np.int16)).to(dev).view(TD[dtype])
    qd = torch.from_numpy(qrows.view(np.int16)).to(dev).view(TD[dtype])
    td = torch.tensor(np.array(tables, np.int32), device=dev)
    ld = torch.tensor(L, dtype=torch.int32, device=dev)
    qq = torch.tensor(qs, device=dev)
    out = torch.empty_like(qd)
    pa.pa_prefill(qd, kc, vc, td, ld, qq, scale, out)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    bound = prefill_weight_bound(qrows, c, tables, L, qs, scale)
    excess = np.abs(got - ref) - half_ulp(np.maximum(np.abs(got), np.abs(ref)), dtype)
    assert excess.max() <= GATE
    assert (excess - U_WEIGHTS[dtype] * bound).max() <= MODEL_SLACK
