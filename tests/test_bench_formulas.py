"""The quantities the roofline figures divide by (CPU).

bench.py reports GB/s of algorithmic bytes for decode and TFLOP/s of causal FLOPs for
prefill; both counts are checked here against a brute-force enumeration of what the
operation reads, writes and multiplies, on small shapes, and against the figures the
measurement notes quote for the bench workloads.
"""

import random

import numpy as np

import bench
import workloads


def _bytes_brute(lens, H, D, B, e):
    # per sequence: every attended token's K and V row of every head, each table entry
    # read (one per frame the sequence occupies), its length; per sequence and head q, out
    total = 0
    for L in lens:
        for _ in range(L):
            total += 2 * H * D * e
        frames = 0
        for t in range(L):
            if t % B == 0:
                frames += 1
        total += 4 * frames + 4
        total += H * D * e * 2
    return total


def _flops_brute(prefix, chunk, H, D):
    total = 0
    for L0, n in zip(prefix, chunk):
        for r in range(n):
            p = L0 + r                       # the query's position
            for _ in range(p + 1):           # keys 0 .. p
                total += H * (2 * D + 2 * D)  # q.k (D multiply-adds), w.v (D multiply-adds)
    return total


def test_algorithmic_bytes_brute_force():
    rnd = random.Random(5)
    for _ in range(20):
        lens = [rnd.randint(0, 70) for _ in range(rnd.randint(1, 6))]
        H, D, B, e = rnd.choice([1, 2, 3]), rnd.choice([8, 16]), rnd.choice([1, 4, 16]), rnd.choice([2, 4])
        assert bench.algorithmic_bytes(lens, H, D, B, e) == _bytes_brute(lens, H, D, B, e)


def test_prefill_flops_brute_force():
    rnd = random.Random(6)
    for _ in range(20):
        k = rnd.randint(1, 4)
        prefix = [rnd.randint(0, 40) for _ in range(k)]
        chunk = [rnd.randint(0, 30) for _ in range(k)]
        H, D = rnd.choice([1, 2]), rnd.choice([4, 8])
        assert bench.prefill_flops(prefix, chunk, H, D) == _flops_brute(prefix, chunk, H, D)


def test_quoted_workload_figures():
    # the chunked-prefill batch: 184.8 GFLOP of causal attention per launch
    w = workloads.prefill_batch()
    (op,) = w.prefill_ops
    seqs, counts = w.ops[op][1], w.ops[op][2]
    prefix = [int(w.final_lens[s]) - int(c) for s, c in zip(seqs, counts)]
    assert round(bench.prefill_flops(prefix, counts, w.num_heads, w.head_dim) / 1e9, 1) == 184.8
    # the decode batch: 1.326 GB of algorithmic bytes for its 64 sequences
    w = workloads.build(1)
    lens = np.array([w.final_lens[s] for s in range(64)])
    assert round(bench.algorithmic_bytes(lens, 32, 128, 16, 2) / 1e9, 3) == 1.326
