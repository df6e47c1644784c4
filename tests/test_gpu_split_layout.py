"""GPU parity of the split cache layout: k [num_blocks, H, D/x, B, x], v
[num_blocks, H, D, B] ("PagedAttention: Virtual Memory Guide for LLM Inference",
"3. PagedAttention CUDA Kernel Execution").

pa_cache_append_split must leave the caches equal, bit for bit, to the oracle's
caches permuted into that layout (oracle.split_layout, pinned on the CPU to the
printed shapes); pa_decode_split must match the oracle's attention element-wise,
with and without context partitions (the merge kernel).
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import replay, split_layout
from tests._gpu_common import assert_attention_close, cache_bits, oracle_bits

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}


def run_split(pa, w):
    dev = torch.device("cuda", 0)
    B, H, D = w.block_size, w.num_heads, w.head_dim
    x = 8
    kc = torch.zeros((w.num_blocks, H, D // x, B * x), dtype=TD[w.dtype], device=dev)
    vc = torch.zeros((w.num_blocks, H, D, B), dtype=TD[w.dtype], device=dev)
    bm = pa.BlockManager(w.num_blocks, B, w.free_order)
    mb = max(1, max(-(-L // B) for L in w.final_lens.values()))
    outs = {}
    for i, op in enumerate(w.ops):
        kind = op[0]
        if kind in ("add", "step", "extend"):
            if kind == "add":
                slots = bm.add_seq(op[1], op[2])
            elif kind == "step":
                slots, copies = bm.step(op[1])
                assert len(copies) == 0
            else:
                slots, copies = bm.extend(op[1], op[2])
                assert len(copies) == 0
            if len(slots):
                k, v = w.rows(i)
                pa.pa_cache_append_split(pa.to_device_rows(k, w.dtype, dev), pa.to_device_rows(v, w.dtype, dev),
                                         torch.from_numpy(np.ascontiguousarray(slots)).to(dev), kc, vc)
        elif kind == "attend":
            tables, lens = bm.block_tables(list(op[1]), mb)
            q = pa.to_device_rows(w.query(i), w.dtype, dev)
            out = torch.empty_like(q)
            pa.pa_decode_split(q, kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                               w.scale, out)
            outs[i] = out
        else:
            raise ValueError(op)
    torch.cuda.synchronize()
    return outs, kc, vc


def check(pa, w):
    outs, kc, vc = run_split(pa, w)
    assert pa.pa_get_device_status() == 0
    ref = replay(w)
    ks, vs = split_layout(ref.cache.k, ref.cache.v, w.elem_bytes)
    assert np.array_equal(cache_bits(kc.view(ks.shape)), oracle_bits(ks))
    assert np.array_equal(cache_bits(vc), oracle_bits(vs))
    for i, out in outs.items():
        assert_attention_close(out, ref.outputs[i], w.dtype)


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_batch(pa, B, dtype):
    rng = np.random.default_rng(B)
    L = rng.integers(1, 700, size=12).tolist() + [0, 1, B - 1, B, B + 1]
    check(pa, workloads.custom(L, H=8, D=128, B=B, dtype=dtype, seed=70 + B))


@pytest.mark.parametrize("B", [8, 16, 32])
def test_head_dim_64(pa, B):
    check(pa, workloads.custom([37, 300, 512, 5], H=4, D=64, B=B, dtype="f16", seed=80 + B))


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("lens", [[2500, 1700], [4096], [255, 256, 257]])
def test_partitions_and_merge(pa, lens, B):
    """Few (sequence, head group) items: the context is split and merged (at B = 32 the
    items hold two heads each, so the partial slots of both group sizes are covered)."""
    check(pa, workloads.custom(lens, H=4, D=128, B=B, dtype="bf16", seed=sum(lens) + B))


def test_rejects_unsupported(pa):
    dev = torch.device("cuda", 0)
    kc = torch.zeros((4, 6, 16, 128), dtype=torch.float16, device=dev)   # H = 6: not a multiple of 4
    vc = torch.zeros((4, 6, 128, 16), dtype=torch.float16, device=dev)
    q = torch.zeros((1, 6, 128), dtype=torch.float16, device=dev)
    t = torch.zeros((1, 2), dtype=torch.int32, device=dev)
    n = torch.ones(1, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PAError) as ei:
        pa.pa_decode_split(q, kc, vc, t, n, 0.1, torch.empty_like(q))
    assert ei.value.code == pa.PA_ERR_UNSUPPORTED
