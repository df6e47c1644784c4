"""No kernel writes outside its outputs (GPU).

With compute-sanitizer closed on this pool, out-of-bounds writes are caught with canary
words instead: every output tensor is a strided view inside a larger buffer -- whole
canary rows before and after it, and a canary gap after every row (the row pitch is
larger than a row) -- and after each call every canary bit must be unchanged.  Each
result is also compared bit for bit with the same call writing a plain contiguous
output, so the strided view is honoured and not just survived.  Covered: pa_decode
(whole sequences, forced partitions with the merge, automatic), the shared-prefix
decode, pa_decode_static, pa_prefill and pa_decode_split.
"""

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

CANARY = 0x7BCD  # a finite fp16 / bf16 bit pattern no kernel computes by chance here
TD = {"f16": torch.float16, "bf16": torch.bfloat16}
PAD, GAP = 3, 64  # canary rows before and after; canary elements after every row


def guarded(n, H, D, dtype):
    """(buffer, view): n rows of [H, D] at row pitch H*D + GAP, PAD canary rows on each side."""
    pitch = H * D + GAP
    buf = torch.empty((n + 2 * PAD) * pitch, dtype=TD[dtype], device="cuda")
    buf.view(torch.int16).fill_(CANARY - 65536 if CANARY > 32767 else CANARY)
    view = buf[PAD * pitch:].as_strided((n, H, D), (pitch, D, 1))
    return buf, view


def assert_guards(buf, n, H, D):
    pitch = H * D + GAP
    bits = buf.view(torch.int16).cpu().numpy().astype(np.int64) & 0xFFFF
    keep = np.ones(bits.shape[0], bool)
    for r in range(n):
        start = (PAD + r) * pitch
        keep[start:start + H * D] = False
    bad = np.nonzero(keep & (bits != CANARY))[0]
    assert bad.size == 0, f"{bad.size} canary elements overwritten, first at offset {bad[:5].tolist()}"


def _inputs(L, H, B, dtype, seed):
    D = 128
    need = sum(-(-x // B) for x in L) + 3
    order = np.random.default_rng(seed).permutation(need)
    tables, pos = [], 0
    mb = max(1, max(-(-x // B) for x in L))
    for x in L:
        n = -(-x // B)
        tables.append(list(order[pos:pos + n]) + [-1] * (mb - n))
        pos += n
    dev = torch.device("cuda")
    kc = torch.from_numpy(workloads.random_storage(seed + 1, (need * B, H, D), dtype).view(np.int16)).to(dev)
    vc = torch.from_numpy(workloads.random_storage(seed + 2, (need * B, H, D), dtype).view(np.int16)).to(dev)
    kc = kc.view(TD[dtype]).view(need, B, H, D)
    vc = vc.view(TD[dtype]).view(need, B, H, D)
    q = torch.from_numpy(workloads.random_storage(seed + 3, (len(L), H, D), dtype).view(np.int16)).to(dev)
    q = q.view(TD[dtype])
    td = torch.tensor(np.array(tables, np.int32), device=dev)
    ld = torch.tensor(L, dtype=torch.int32, device=dev)
    return kc, vc, q, td, ld


@pytest.mark.parametrize("params", [{"partition_tokens": -1}, {"partition_tokens": 32}, {},
                                    {"share_prefix": 16}, "static"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_writes_only_its_rows(pa, params, dtype):
    B, H = 16, 4
    L = [1, 15, 16, 17, 300, 777, 0, 64]
    kc, vc, q, td, ld = _inputs(L, H, B, dtype, seed=5)
    if params == {"share_prefix": 16}:  # neighbours that share their leading frames
        td[1, :2] = td[0, :2]
        td[5, :18] = td[4, :18]
        ld[5] = 300
    n, D = len(L), 128
    buf, out = guarded(n, H, D, dtype)
    ref = torch.empty((n, H, D), dtype=TD[dtype], device="cuda")
    if params == "static":
        pa.pa_decode_static(q, kc, vc, td, ld, 0.0883883, out)
        pa.pa_decode_static(q, kc, vc, td, ld, 0.0883883, ref)
    else:
        pa.pa_decode_ex(q, kc, vc, td, ld, 0.0883883, out, params)
        pa.pa_decode_ex(q, kc, vc, td, ld, 0.0883883, ref, params)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    assert_guards(buf, n, H, D)
    assert torch.equal(out.contiguous().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_writes_only_its_rows(pa, dtype):
    B, H, D = 16, 4, 128
    L = [40, 300, 129, 513]
    counts = [40, 130, 1, 257]
    kc, vc, _, td, ld = _inputs(L, H, B, dtype, seed=9)
    T = sum(counts)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    q = torch.from_numpy(workloads.random_storage(11, (T, H, D), dtype).view(np.int16)).to("cuda").view(TD[dtype])
    buf, out = guarded(T, H, D, dtype)
    ref = torch.empty((T, H, D), dtype=TD[dtype], device="cuda")
    pa.pa_prefill(q, kc, vc, td, ld, qs, 0.0883883, out)
    pa.pa_prefill(q, kc, vc, td, ld, qs, 0.0883883, ref)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    assert_guards(buf, T, H, D)
    assert torch.equal(out.contiguous().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("L", [[5, 300, 1200, 16], [4000, 3000]])
def test_split_layout_decode_writes_only_its_rows(pa, L):
    B, H, D, dtype = 16, 8, 128, "f16"
    kc, vc, q, td, ld = _inputs(L, H, B, dtype, seed=13)
    nb = kc.shape[0]
    ks = kc.view(nb, B, H, D // 8, 8).permute(0, 2, 3, 1, 4).contiguous().view(nb, H, D // 8, B * 8)
    vs = vc.permute(0, 2, 3, 1).contiguous()
    n = len(L)
    buf, out = guarded(n, H, D, dtype)
    ref = torch.empty((n, H, D), dtype=TD[dtype], device="cuda")
    pa.pa_decode_split(q, ks, vs, td, ld, 0.0883883, out)
    pa.pa_decode_split(q, ks, vs, td, ld, 0.0883883, ref)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    assert_guards(buf, n, H, D)
    assert torch.equal(out.contiguous().view(torch.int16), ref.view(torch.int16))
