"""pa_decode_static: decode attention that allocates no device memory (GPU).

Some callers cannot let a library call cudaMalloc: a serving process whose
device memory is owned by its own pool allocator, or a latency-bound loop that
cannot take the device-wide synchronisation of a first allocation.  For them
pa_decode_static takes its scratch from a fixed 16 MiB array compiled into
libpa.  These tests call it through the C ABI and compare it with the fp64 oracle
and with pa_decode on the same inputs, on two calls in a row (the array keeps the
previous call's contents); check that a call on a stream the library has never
seen leaves the device's free memory unchanged (where pa_decode would allocate
its workspace); and check that a problem needing more scratch than the array
holds is refused without launching anything.

This file is collected last on purpose: it should pass alone in a fresh process
and after every other test.
"""

import pytest
import torch

import workloads
from oracle import replay
from tests._gpu_common import assert_attention_close

pytestmark = pytest.mark.gpu


def _engine_batch(pa, w):
    eng = pa.PagedKVEngine(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype,
                           free_order=w.free_order, max_seqs=max(64, len(w.final_lens)),
                           max_blocks_per_seq=max(1, max(-(-L // w.block_size) for L in w.final_lens.values())))
    pa.run_workload_ops(eng, w)
    (op,) = w.attend_ops
    seqs = w.ops[op][1]
    tables, lens = eng.bm.block_tables(seqs, eng.max_blocks)
    q = pa.to_device_rows(w.query(op), w.dtype, eng.device)
    return eng, q, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()


@pytest.mark.parametrize("lengths,H,B,dtype", [
    ([300, 1000, 17, 4000, 2048, 0, 1, 16], 8, 16, "f16"),   # split contexts + merge, unrolled path
    ([2500, 5, 700, 33], 4, 32, "bf16"),                     # two warps per head
    ([9, 130, 41], 3, 10, "f32"),                            # generic path, B not a power of two
])
def test_static_scratch_matches_oracle_and_pa_decode(pa, lengths, H, B, dtype):
    w = workloads.custom(lengths, H=H, D=128 if dtype != "f32" else 64, B=B, dtype=dtype, seed=77)
    eng, q, tables, lens = _engine_batch(pa, w)
    (op,) = w.attend_ops
    oracle = replay(w).outputs[op]
    ref = torch.empty_like(q)
    pa.pa_decode(q, eng.k_cache, eng.v_cache, tables, lens, w.scale, ref)
    torch.cuda.synchronize()
    ref64 = ref.double().cpu().numpy()
    assert_attention_close(ref, oracle, dtype)
    for _ in range(2):  # the second call starts from the first call's leftovers
        out = torch.full_like(q, float("nan"))
        pa.pa_decode_static(q, eng.k_cache, eng.v_cache, tables, lens, w.scale, out)
        torch.cuda.synchronize()
        assert_attention_close(out, oracle, dtype)
        assert_attention_close(out, ref64, dtype)
    assert pa.pa_get_device_status() == 0


def test_static_scratch_allocates_nothing(pa):
    """A call on a stream the library has never seen (pa_decode would allocate a
    workspace for it) leaves the device's free memory as it was; pa_decode on another
    new stream, for contrast, takes some."""
    w = workloads.custom([4000, 300, 2048, 17, 1200, 9000], H=8, D=128, B=16, dtype="f16", seed=78)
    eng, q, tables, lens = _engine_batch(pa, w)
    (op,) = w.attend_ops
    oracle = replay(w).outputs[op]
    out = torch.full_like(q, float("nan"))
    out2 = torch.full_like(q, float("nan"))
    # a first call loads the library's device code and its fixed array (module load,
    # not an allocation by the call)
    pa.pa_decode_static(q, eng.k_cache, eng.v_cache, tables, lens, w.scale, out2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s1):
        pa.pa_decode_static(q, eng.k_cache, eng.v_cache, tables, lens, w.scale, out)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"pa_decode_static changed free device memory by {free0 - free1} bytes"
    assert_attention_close(out, oracle, "f16")
    with torch.cuda.stream(s2):
        pa.pa_decode(q, eng.k_cache, eng.v_cache, tables, lens, w.scale, out2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free1, "the free-memory probe did not see pa_decode's workspace"
    assert_attention_close(out2, oracle, "f16")
    assert pa.pa_get_device_status() == 0


def test_static_scratch_refuses_oversized_problem(pa):
    S, H, D, B, nb, mb = 4096, 32, 128, 16, 64, 20   # needs ~70 MB of split partials
    kc = torch.zeros(nb, B, H, D, dtype=torch.float16, device="cuda")
    q = torch.zeros(S, H, D, dtype=torch.float16, device="cuda")
    out = torch.full_like(q, 3.0)
    tables = torch.zeros(S, mb, dtype=torch.int32, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    n0 = pa.pa_launch_count()
    with pytest.raises(pa.PAError) as ei:
        pa.pa_decode_static(q, kc, kc, tables, lens, 0.1, out)
    assert ei.value.code == pa.PA_ERR_SCRATCH_LIMIT
    assert pa.pa_launch_count() == n0
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
