#!/usr/bin/env python
"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of a 64-sequence batch through libpa: host block
manager step (slots, copy-on-write pairs, block tables) -> one staged upload ->
pa_cache_append of the 64 new K/V rows -> pa_decode (+ merge).  The workload is
the decode batch of 64 sequences with context lengths ~U[512, 2048], 32 heads,
head_dim 128, block_size 16, fp16 K/V/q, physical frames handed out in shuffled
order from a pool 1.2x the need.

The bench keeps R independent copies of that batch resident and decodes them in
rotation, so every step reads a different ~1.3 GB batch (far beyond the 129 MB
L2: no flush needed) and each batch's lengths drift only K/R tokens over the run;
prefill lengths are centred so that the mean attended length over the timed
steps equals the sampled length.

Printed: one JSON line (rank 0) with the throughput of the whole step (value:
the K timed steps, nothing else on the stream), the decode kernel's roofline
figure (pa_decode alone, timed in a separate phase after the steps: back-to-back
launches over the resident batches), the end-to-end figure through host buffers,
the other serving shapes and the chunked prefill under ``extra``, the oracle's
CPU baseline (one thread, and one worker per affine core), launch count and SM
clocks sampled while the GPU works.  ``--impl reference`` times the CPU oracle
instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV bytes GB/s (% of GB300 HBM peak); seqs/sec at 64×2k"
UNIT = "GB/s"


def algorithmic_bytes(lens, H, D, B, e_kv, e_q=None, e_out=None) -> int:
    """K and V rows of every attended token, the block-table entries read, the
    context lengths, q and out.  Tail padding of the last frame and split
    workspace traffic are not counted."""
    e_q = e_kv if e_q is None else e_q
    e_out = e_kv if e_out is None else e_out
    total = 0
    for L in lens:
        L = int(L)
        total += 2 * L * H * D * e_kv + 4 * (-(-L // B))
    S = len(lens)
    return total + 4 * S + S * H * D * (e_q + e_out)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def _kernel_source_hash() -> str:
    """Hash of the decode kernel's device code (decode_kernel.cuh up to its host-side
    launchers): DRAM bytes per launch are the kernel's, not the launch code's."""
    with open(os.path.join(ROOT, "paged_kv_cache_126_gb300", "csrc", "decode_kernel.cuh"), "rb") as fh:
        src = fh.read()
    cut = src.find(b"// ---- host-side launcher")
    return hashlib.sha256(src[:cut] if cut >= 0 else src).hexdigest()[:12]


def _profile_traffic(workload_key: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_decode_batch_64.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_src = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    m_tr = re.search(rf"traffic_bytes_per_launch\[{re.escape(workload_key)}\]:\s*([0-9.eE+]+)", txt)
    if not m_src or not m_tr or m_src.group(1) != _kernel_source_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu, self.interval, self.proc, self.out = str(gpu_index), interval_ms, None, ""
        try:  # the CUDA ordinal need not match nvidia-smi's index; the UUID does
            import torch
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.interval}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_sample(cfg, n_seqs, seed_shift=0):
    """A few sequences of the bench workload with host data, replayed by the oracle."""
    import numpy as np

    import workloads
    from oracle import replay

    w = workloads.build(cfg)
    rng = np.random.default_rng(99 + seed_shift)
    keep = sorted(rng.choice(len(w.final_lens), n_seqs, replace=False).tolist())
    ref = replay(w, keep_seqs=keep, with_cache=True)
    op = w.attend_ops[-1]
    q = w.query(op)
    tables, lens = ref.attend_meta[op]
    return w, ref, keep, q[keep], [tables[j] for j in keep], [lens[j] for j in keep]


def cpu_baseline_worker(cfg, budget_s: float, per_step: bool = False, steps: int = 0, seed_shift: int = 0):
    """Time the oracle's paged decode (gather + fp64 softmax attention) on host cores."""
    from oracle import paged_decode

    # the toy has 4 sequences; a long-context sequence (16384 tokens) is a sample by itself
    n = 1 if cfg == 2 else (4 if (not per_step or cfg == 0) else 8)
    w, ref, keep, q, tables, lens = _oracle_sample(cfg, n, seed_shift)
    bytes_per_seq = [algorithmic_bytes([L], w.num_heads, w.head_dim, w.block_size, w.elem_bytes) for L in lens]
    if per_step:
        times, byts = [], []
        for k in range(steps):
            j = k % len(keep)
            t0 = time.perf_counter()
            paged_decode(q[j:j + 1], ref.cache, [tables[j]], [lens[j]], w.scale)
            times.append(time.perf_counter() - t0)
            byts.append(bytes_per_seq[j])
        return {"times": times, "bytes": byts, "sample": f"1 of {len(keep)} sampled sequences per step "
                                                         f"(lengths {lens}), {w.num_heads} heads"}
    done, elapsed, nbytes = 0, 0.0, 0
    while elapsed < budget_s:
        j = done % len(keep)
        t0 = time.perf_counter()
        paged_decode(q[j:j + 1], ref.cache, [tables[j]], [lens[j]], w.scale)
        elapsed += time.perf_counter() - t0
        nbytes += bytes_per_seq[j]
        done += 1
    return {"value": nbytes / elapsed / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} single-sequence oracle decodes cycling over {len(keep)} sampled sequences "
                      f"(lengths {lens}) of the bench workload, {elapsed:.1f} s, one thread",
            "seqs_per_sec": done / elapsed}


_CPU_ENV = dict(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")


def _cpu_cmd(cfg, budget_s, seed_shift=0):
    return [sys.executable, os.path.abspath(__file__), "--cpu-worker", str(cfg), "--cpu-budget", str(budget_s),
            "--cpu-seed-shift", str(seed_shift)]


def run_cpu_baseline(cfg, budget_s: float):
    env = dict(os.environ, **_CPU_ENV)
    res = subprocess.run(_cpu_cmd(cfg, budget_s), capture_output=True, text=True, env=env,
                         timeout=max(600, 20 * budget_s))
    if res.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "error": res.stderr[-400:]}
    return json.loads(res.stdout.strip().splitlines()[-1])


def run_cpu_all_cores(cfg, budget_s: float):
    """One single-threaded oracle worker per affine core, all at once, each on its own
    sampled sequences for ``budget_s`` seconds of decode time; the rates add up."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    env = dict(os.environ, **_CPU_ENV)
    procs = [subprocess.Popen(_cpu_cmd(cfg, budget_s, 1 + i), stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True, env=env) for i in range(cores)]
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=max(900, 30 * budget_s))
        if p.returncode != 0:
            return {"value": None, "cores": cores, "error": e[-400:]}
        outs.append(json.loads(o.strip().splitlines()[-1]))
    sps = sum(o["seqs_per_sec"] for o in outs)
    return {"value": sum(o["value"] for o in outs), "unit": UNIT, "cores": cores, "seqs_per_sec": sps,
            "s_per_call": 1.0 / sps,
            "sample": f"{cores} single-threaded workers at once, each cycling over its own sampled "
                      f"sequences for {budget_s:.0f} s of decode time"}


def cpu_sweep(keys=("0", "1", "2", "3", "4"), budget_s: float = 8.0):
    """The oracle's decode timed on the host per workload: one thread, then one
    single-threaded worker per affine core at once (each on its own sampled sequences);
    one JSON line per workload."""
    for key in keys:
        single = run_cpu_baseline(key, budget_s)
        allc = run_cpu_all_cores(key, budget_s)
        if allc["value"] is None:
            raise SystemExit(f"cpu worker failed: {allc['error']}")
        print(json.dumps({
            "cpu_baseline": key, "kind": "oracle", "unit": UNIT,
            "single": {"cores": 1, "gbps": round(single["value"], 3), "seqs_per_sec": round(single["seqs_per_sec"], 2),
                       "s_per_call": round(1.0 / single["seqs_per_sec"], 5), "sample": single["sample"]},
            "all_cores": {"cores": allc["cores"], "gbps": round(allc["value"], 3),
                          "seqs_per_sec": round(allc["seqs_per_sec"], 2), "s_per_call": round(allc["s_per_call"], 6),
                          "sample": allc["sample"]},
            "call": "one single-sequence decode (all heads): gather of the sequence's frames, fp64 attention"}),
            flush=True)


# ----------------------------------------------------------------------------- GPU arm
def _dist_init():
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def reduce_max_sum(max_val: float, sum_val: float, device=None):
    """(max over ranks of max_val, sum over ranks of sum_val); identity at world 1."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return max_val, sum_val
    t = torch.tensor([max_val], dtype=torch.float64, device=device)
    u = torch.tensor([sum_val], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist

    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own batches (weak scaling by sequences)."""
    return base + 7919 * rank


class DecodeBench:
    """R resident copies of the decode batch on one device, decoded in rotation."""

    def __init__(self, cfg, R, steps_per_batch_max, centre_steps, seed, device):
        import numpy as np
        import torch

        import paged_kv_cache_126_gb300 as pa
        import workloads

        self.pa, self.torch = pa, torch
        w = workloads.build(cfg)
        self.w = w
        S = len(w.final_lens)
        self.S, self.H, self.D, self.B = S, w.num_heads, w.head_dim, w.block_size
        self.e = w.elem_bytes
        self.R = R
        L = np.array([w.final_lens[s] for s in range(S)], dtype=np.int64)
        self.L = L
        prefill = np.maximum(L - 1 - centre_steps, 0)
        final = prefill + steps_per_batch_max
        need = int(sum(-(-int(x) // self.B) for x in final)) * R
        nb = int(math.ceil(1.2 * need)) + R * S
        rng = np.random.default_rng(seed)
        order = rng.permutation(nb).astype(np.int32)
        max_blocks = int(-(-int(final.max()) // self.B)) + 1
        self.eng = pa.PagedKVEngine(nb, self.B, self.H, self.D, w.dtype, free_order=order, device=device,
                                    max_seqs=S, max_blocks_per_seq=max_blocks)
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        dt = pa.engine.TORCH_DTYPES[w.dtype]
        self.batches = []
        for r in range(R):
            ids = list(range(r * S, (r + 1) * S))
            for j, s in enumerate(ids):
                n = int(prefill[j])
                k = torch.randn(n, self.H, self.D, generator=g, device=device).to(dt)
                v = torch.randn(n, self.H, self.D, generator=g, device=device).to(dt)
                self.eng.add_seq(s, k, v)
            self.batches.append(ids)
        self.inputs = []
        for _ in range(4):
            mk = lambda: torch.randn(S, self.H, self.D, generator=g, device=device).to(dt)  # noqa: E731
            self.inputs.append((mk(), mk(), mk()))
        self.out = torch.empty(S, self.H, self.D, dtype=dt, device=device)
        self.scale = w.scale
        torch.cuda.synchronize()

    def step(self, k):
        kn, vn, q = self.inputs[k % 4]
        out, nc, lens = self.eng.decode_step(self.batches[k % self.R], kn, vn, q, self.scale, self.out)
        return algorithmic_bytes(lens, self.H, self.D, self.B, self.e), lens

    def decode_only(self, n):
        """pa_decode alone: n back-to-back launches over the resident batches in rotation
        (every launch reads a different batch, far beyond L2), each batch at its current
        length.  The launches are queued behind a ~1 ms GPU sleep, so the start event
        fires with launches already waiting and no host enqueue time falls inside the
        bracket.  Returns (mean us per launch, mean algorithmic bytes per launch, n)."""
        torch = self.torch
        st = torch.cuda.current_stream(self.eng.device)
        metas = []
        for ids in self.batches:
            tables, lens = self.eng.bm.block_tables(ids, self.eng.max_blocks)
            metas.append((torch.from_numpy(tables).to(self.eng.device), torch.from_numpy(lens).to(self.eng.device),
                          algorithmic_bytes(lens, self.H, self.D, self.B, self.e)))
        q = self.inputs[0][2]
        out = torch.empty_like(self.out)
        kc, vc = self.eng.k_cache, self.eng.v_cache

        def launch(i):
            t, ln, _ = metas[i % self.R]
            self.pa.pa_decode(q, kc, vc, t, ln, self.scale, out)

        for i in range(3):
            launch(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)
        e0.record(st)
        for i in range(n):
            launch(i)
        e1.record(st)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n
        return us, sum(metas[i % self.R][2] for i in range(n)) / n, n


def gpu_arm(args):
    import numpy as np
    import torch

    rank, local, world = _dist_init()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import paged_kv_cache_126_gb300 as pa

    K, W = args.steps, args.warmup
    R = args.batches
    k_e2e = max(args.e2e_steps, R)
    per_batch = -(-(W + K + k_e2e) // R) + 2
    centre = -(-W // R) + (K // R + 1) // 2
    bench = DecodeBench(args.config, R, per_batch, centre, rank_seed(1234, rank), device)
    st = torch.cuda.current_stream(device)

    # The clock sampler starts before the warm-up: its start-up must not leave the GPU
    # idle between the warm-up and the timed steps.
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier()
    for k in range(W):
        bench.step(k)
    torch.cuda.synchronize()

    # ---- timed region: K whole steps (pa_step_decode), inputs resident in HBM ----------------
    # Nothing but the steps runs on the stream between the two events.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    n_launch0 = pa.pa_launch_count()
    step_bytes, all_lens = [], []
    t_start.record(st)
    for k in range(K):
        b, lens = bench.step(W + k)
        step_bytes.append(b)
        all_lens.append(float(np.mean(lens)))
    t_end.record(st)
    torch.cuda.synchronize()
    barrier()
    launches = pa.pa_launch_count() - n_launch0
    ms = t_start.elapsed_time(t_end)
    my_bytes = float(sum(step_bytes))
    max_ms, tot_bytes = reduce_max_sum(ms, my_bytes, device)

    # ---- the decode kernel alone (roofline), after the timed region --------------------------
    n_dec = max(32, 2 * R)
    dec_us, dec_bytes, _ = bench.decode_only(n_dec)
    clk = clocks.stop() if rank == 0 else None

    # ---- end to end: host buffers, copies inside the timed region ---------------------------
    dt = bench.inputs[0][0].dtype
    S, H, D = bench.S, bench.H, bench.D
    # Every step copies its k/v/q rows in from pinned host memory and its output back.  The
    # copies run on a copy stream, pipelined a group of G steps ahead over 2G buffers: the
    # inputs of the next group travel while this group computes, and each output goes back
    # as soon as its step is done.  The compute stream waits on the copy stream once per
    # group (a wait between two kernels costs the programmatic launch overlap of that pair).
    host_in = [tuple(x.cpu().pin_memory() for x in trip) for trip in bench.inputs]
    G = 4
    nbuf = 2 * G
    dev_in = [[torch.empty(S, H, D, dtype=dt, device=device) for _ in range(3)] for _ in range(nbuf)]
    dev_out = [torch.empty(S, H, D, dtype=dt, device=device) for _ in range(nbuf)]
    host_out = [torch.empty(S, H, D, dtype=dt).pin_memory() for _ in range(nbuf)]
    cs = torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # the inputs of step k (buffer k mod nbuf) have landed
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]  # step k has finished
    ev_read = [torch.cuda.Event() for _ in range(nbuf)]  # step k's output has reached the host
    mb = bench.eng.max_blocks
    h2d = 3 * S * H * D * bench.e + 4 * (4 * S + S * mb)
    d2h = S * H * D * bench.e

    def load_group(k0):
        """Inputs of steps k0 .. k0 + G - 1 (their buffers last served steps k0 - nbuf ..)."""
        with torch.cuda.stream(cs):
            if k0 >= nbuf:
                cs.wait_event(ev_done[(k0 - nbuf + G - 1) % nbuf])
            for k in range(k0, min(k0 + G, k_e2e)):
                for x, hx in zip(dev_in[k % nbuf], host_in[k % 4]):
                    x.copy_(hx, non_blocking=True)
                ev_in[k % nbuf].record(cs)

    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = 0
    e0.record(st)
    cs.wait_event(e0)
    load_group(0)
    for k in range(k_e2e):
        b = k % nbuf
        if k % G == 0:
            if k + G < k_e2e:
                load_group(k + G)
            # this group's inputs, and its output buffers free (their outputs, G steps and
            # more before, read back)
            st.wait_event(ev_in[(min(k + G, k_e2e) - 1) % nbuf])
            if k >= nbuf:
                st.wait_event(ev_read[(k + G - 1 - nbuf) % nbuf])
        out, _, lens = bench.eng.decode_step(bench.batches[(W + K + k) % R], dev_in[b][0], dev_in[b][1],
                                             dev_in[b][2], bench.scale, dev_out[b])
        ev_done[b].record(st)
        e2e_bytes += algorithmic_bytes(lens, H, D, bench.B, bench.e)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[b])
            host_out[b].copy_(out, non_blocking=True)
            ev_read[b].record(cs)
    st.wait_stream(cs)
    e1.record(st)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    e2e_max_ms, e2e_tot = reduce_max_sum(e2e_ms, float(e2e_bytes), device)

    if rank != 0:
        return
    peak, peak_src = _peaks()
    achieved = dec_bytes / (dec_us * 1e-6) / 1e9
    traffic = _profile_traffic("decode batch 64 x U[512,2048]")
    value = tot_bytes / (max_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(max_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded; K/V/q ~ N(0,1) fp16; lengths and shuffled free order from the workload generator)",
        "config": {
            "workload": "decode batch: 64 seqs, context ~U[512,2048], 32 heads, head_dim 128, block_size 16, fp16",
            "seqs_per_step": S,
            "mean_attended_len": round(float(np.mean(all_lens)), 1),
            "sampled_mean_len": round(float(bench.L.mean()), 1),
            "resident_batches": R,
            "l2": f"inputs larger than L2: each step reads a different ~{my_bytes / K / 1e9:.2f} GB batch",
            "parallelism": f"replicas by sequence batch x{world}",
        },
        "seqs_per_sec": round(S * K * world / (max_ms * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "decode_kernel (pa_decode; the log-sum-exp merge runs inside it)",
            "timing": f"CUDA events around {n_dec} back-to-back pa_decode launches over the {R} resident "
                      f"batches in rotation (each launch reads a different batch, > L2), queued behind a GPU sleep; "
                      f"run after the timed steps",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_source": peak_src,
            "decode_us_per_launch": round(dec_us, 2),
            "algorithmic_bytes_per_launch": round(dec_bytes),
            "launches": n_dec,
            "decode_within_step": bool(dec_us <= 1000 * max_ms / K),
        },
        "e2e": {
            "value": round(e2e_tot / (e2e_max_ms * 1e-3) / 1e9, 1),
            "unit": UNIT,
            "steps": k_e2e,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "api": "PagedKVEngine.decode_step with q/k/v copied from pinned host buffers and out copied back "
                   "every step (copies on a second stream, pipelined a group of four steps ahead)",
        },
        "gpu_launches": launches,
        "clocks": clk,
    }
    if not args.no_extra:
        del bench
        torch.cuda.empty_cache()
        line["extra"] = {"fixed_64x2048": _guarded(lambda: fixed_variant(args, device)), **bench_extras(device)}
    if not args.no_cpu:
        cpu = run_cpu_baseline(args.config, args.cpu_budget or 8.0)
        allc = run_cpu_all_cores(args.config, args.cpu_budget or 8.0)
        if allc.get("value") is not None:
            allc["value"] = round(allc["value"], 3)
        cpu["all_cores"] = allc
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def _guarded(fn):
    """fn(), or its error in one line: a failing extra figure must not lose the line."""
    try:
        return fn()
    except Exception as e:  # noqa: BLE001
        return {"error": f"{type(e).__name__}: {e}"[:300]}


def fixed_variant(args, device):
    """The same step on 64 sequences of exactly 2048 tokens (the '64x2k' figure), then
    the decode kernel alone as in the main line."""
    import torch

    R, K = 4, max(40, args.steps // 8)
    bench = DecodeBench("1x", R, -(-(K + 8) // R) + 2, 2 + (K // R + 1) // 2, 4321, device)
    st = torch.cuda.current_stream(device)
    for k in range(8):
        bench.step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0
    e0.record(st)
    for k in range(K):
        b, _ = bench.step(8 + k)
        tot += b
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    dec_us, dec_bytes, n_dec = bench.decode_only(32)
    peak, _ = _peaks()
    res = {"steps": K, "gbps": round(tot / (ms * 1e-3) / 1e9, 1), "seqs_per_sec": round(64 * K / (ms * 1e-3), 1),
           "ms_per_step": round(ms / K, 5),
           "decode_us_per_launch": round(dec_us, 2), "decode_launches": n_dec,
           "decode_gbps": round(dec_bytes / (dec_us * 1e-6) / 1e9, 1),
           "decode_frac": round(dec_bytes / (dec_us * 1e-6) / 1e9 / peak, 4),
           "decode_seqs_per_sec": round(64 / (dec_us * 1e-6), 1)}
    del bench
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- per-workload sweep
SWEEP_KEYS = ("0", "1", "1x", "2", "2n", "3", "3c", "3s", "4")


def replay_device_rows(eng, w, seed):
    """Run a workload's operations through the engine with the K/V rows drawn on the
    device: the workload's lengths, forks, copy-on-write copies, frees and frame order,
    values N(0, sigma^2) rounded to the storage dtype.  For timing only (the values do
    not change the work); drawing multi-GB caches on the host would dominate the run.
    Returns the number of copy-on-write frame copies."""
    import torch

    import paged_kv_cache_126_gb300 as pa

    g = torch.Generator(device=eng.device)
    g.manual_seed(seed)
    dt = pa.engine.TORCH_DTYPES[w.dtype]
    H, D = w.num_heads, w.head_dim

    def rows(n):
        mk = lambda: (torch.randn(n, H, D, generator=g, device=eng.device) * w.sigma).to(dt)  # noqa: E731
        return mk(), mk()

    copies = 0
    for op in w.ops:
        kind = op[0]
        if kind == "add":
            eng.add_seq(op[1], *rows(op[2]))
        elif kind == "fork":
            eng.fork(op[1], op[2])
        elif kind == "step":
            copies += len(eng.step(op[1], *rows(len(op[1])))[1])
        elif kind == "extend":
            copies += len(eng.extend(op[1], *rows(op[2]))[1])
        elif kind == "free":
            eng.free(op[1])
        elif kind not in ("attend", "prefill"):
            raise ValueError(f"op {kind!r} has no device-row replay")
    return copies


def _workload_engine(key, dev, device_rows):
    """Engine holding workload `key` at its final state (host-drawn rows through the
    workload generator, or device-drawn rows), plus the copy-on-write copy count."""
    import paged_kv_cache_126_gb300 as pa
    import workloads

    cfg = {"0": 0, "1": 1, "1x": "1x", "2": 2, "2n": 2, "3": 3, "3c": 3, "3s": 3, "4": 4, "4d": 4}[key]
    w = workloads.build(cfg)
    if key == "4d":
        # the serving mix scaled down for a profiler capture: its first 48 of 256 sequences
        # (same length law, 40 heads, bf16 N(0, 0.5), prefill L-1 + one appended token)
        L = [w.final_lens[s] for s in range(48)]
        w = workloads.custom(L, H=w.num_heads, D=w.head_dim, B=w.block_size, dtype=w.dtype, sigma=w.sigma,
                             seed=w.seed, name="serving mix, first 48 of 256 seqs: L~logU[16,8192], H=40, D=128, "
                                               "B=16, bf16")
    if key == "3c":
        L = [w.final_lens[s] for s in range(len(w.final_lens))]
        w = workloads.custom(L, H=w.num_heads, D=w.head_dim, B=w.block_size, dtype=w.dtype, seed=w.seed,
                             name="parallel-sampling control: same lengths, no shared frames")
    eng = pa.PagedKVEngine(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype,
                           free_order=w.free_order, device=dev, max_seqs=max(64, len(w.final_lens)),
                           max_blocks_per_seq=max(1, max(-(-L // w.block_size) for L in w.final_lens.values())))
    if device_rows:
        copies = replay_device_rows(eng, w, 4000 + w.seed)
    else:
        _, trace = pa.run_workload_ops(eng, w)
        copies = sum(len(t["copies"]) for t in trace.values() if isinstance(t, dict) and "copies" in t)
    return w, eng, copies


def decode_figures(key, reps=20, flushed_reps=50, device_rows=False, memset=True, append=True,
                   sample_clocks=False):
    """pa_decode on the final state of one workload's replay (automatic launch options;
    "3s": the engine's automatic choice, the shared-prefix decode; "2n": no
    split-context partitions), timed two ways.

    ``decode_us``: mean over ``reps`` back-to-back launches queued behind a GPU sleep.
    ``flushed``: median over ``flushed_reps`` launches each timed alone with CUDA events
    after a read of twice the L2 size (no K/V byte served from L2 left warm by the
    previous launch).  A read leaves clean lines; a memset flush (``flushed_memset``)
    leaves the L2 full of dirty lines whose write-back (~the L2 size) then lands inside
    the timed launch.  Bytes: algorithmic (logical: every sequence's attended tokens)
    and unique frames (each frame that some sequence reads, once)."""
    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa

    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    w, eng, copies = _workload_engine(key, dev, device_rows)
    op = w.attend_ops[-1]
    seqs = w.ops[op][1]
    tables, lens = eng.bm.block_tables(seqs, eng.max_blocks)
    if key == "3s":
        params = eng._decode_params(tables, None)
        assert params is not None, "the parallel-sampling batch should take the shared-prefix decode"
    else:
        params = {"partition_tokens": -1} if key == "2n" else None
    tt, ll = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    q = pa.to_device_rows(w.query(op), w.dtype, dev)
    out = torch.empty_like(q)

    def decode():
        pa.pa_decode(q, eng.k_cache, eng.v_cache, tt, ll, w.scale, out, params=params)

    clocks = ClockSampler(dev.index, interval_ms=20) if sample_clocks else None
    if clocks:
        clocks.start()
    for _ in range(3):
        decode()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(2_000_000)
    e0.record(st)
    for _ in range(reps):
        decode()
    e1.record(st)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 132 * 2 ** 20
    flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(flushed_reps)]

    def isolated(fn, clear):
        for a, b in ev:
            clear()
            a.record(st)
            fn()
            b.record(st)
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e3

    us_flushed = isolated(decode, lambda: flush.sum())
    clk = clocks.stop() if clocks else None
    us_memset = isolated(decode, lambda: flush.zero_()) if memset else None
    logical = algorithmic_bytes(lens, w.num_heads, w.head_dim, w.block_size, w.elem_bytes)
    frames = set()
    for t, L in zip(tables, lens):
        frames.update(t[: -(-int(L) // w.block_size)].tolist())
    unique = len(frames) * w.block_size * w.num_heads * w.head_dim * w.elem_bytes * 2
    peak, _ = _peaks()
    gb = lambda b, t: round(b / (t * 1e-6) / 1e9, 1)  # noqa: E731
    res = {
        "workload": key, "name": w.name, "params": params, "seqs": len(seqs), "sum_len": int(np.sum(lens)),
        "data": "device-drawn rows (timing only)" if device_rows else "host-drawn rows (the workload generator)",
        "decode_us": round(us, 2), "algorithmic_bytes": logical, "gbps": gb(logical, us),
        "pct_of_peak": round(100 * logical / (us * 1e-6) / 1e9 / peak, 1),
        "unique_frame_bytes": unique, "gbps_unique_frames": gb(unique, us),
        "seqs_per_sec": round(len(seqs) / (us * 1e-6), 1),
        "flushed": {"decode_us_median": round(us_flushed, 2), "launches": flushed_reps,
                    "gbps": gb(logical, us_flushed),
                    "pct_of_peak": round(100 * logical / (us_flushed * 1e-6) / 1e9 / peak, 1),
                    "gbps_unique_frames": gb(unique, us_flushed),
                    "frac_unique_frames": round(unique / (us_flushed * 1e-6) / 1e9 / peak, 4),
                    "seqs_per_sec": round(len(seqs) / (us_flushed * 1e-6), 1)},
        "cow_copies": copies,
    }
    if us_memset is not None:
        res["flushed_memset"] = {"decode_us_median": round(us_memset, 2), "gbps": gb(logical, us_memset)}
    if clk is not None:
        res["clocks"] = clk
    if append:
        # pa_cache_append of one new row per sequence at its last token's slot (the rows
        # already there, so the cache is unchanged): read k_new, v_new and the slots,
        # write the two cache rows
        slots = torch.tensor([eng.bm.slot(s, int(L) - 1) for s, L in zip(seqs, lens) if L > 0],
                             dtype=torch.int32, device=dev)
        kn = eng.k_cache.view(-1, w.num_heads, w.head_dim)[slots.long()].contiguous()
        vn = eng.v_cache.view(-1, w.num_heads, w.head_dim)[slots.long()].contiguous()

        def app():
            pa.pa_cache_append(kn, vn, slots, eng.k_cache, eng.v_cache)

        for _ in range(3):
            app()
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(reps):
            app()
        e1.record(st)
        torch.cuda.synchronize()
        ap_us = e0.elapsed_time(e1) / reps * 1e3
        ap_us_flushed = isolated(app, lambda: flush.sum())
        ap_bytes = 4 * kn.numel() * kn.element_size() + 4 * slots.numel()
        res["append"] = {"rows": int(slots.numel()), "bytes": int(ap_bytes), "us": round(ap_us, 2),
                         "gbps": gb(ap_bytes, ap_us), "us_flushed_median": round(ap_us_flushed, 2),
                         "gbps_flushed": gb(ap_bytes, ap_us_flushed)}
    del flush, eng, tt, ll, q, out
    torch.cuda.empty_cache()
    return res


def sweep(keys, reps=20, flushed_reps=50):
    """pa_decode on the final state of each workload's replay (host-drawn rows): one
    JSON line per workload (``decode_figures``).  "3c" is the unshared control of the
    parallel-sampling workload (the same final lengths, every branch with private
    frames); "3s" is the parallel-sampling workload through the shared-prefix decode
    (each shared prompt frame read once for its branches); "2n" is the long-context
    workload without split-context partitions (one item per sequence and head group),
    the baseline of the split's speedup."""
    import torch

    torch.cuda.set_device(0)
    for key in keys:
        print(json.dumps(decode_figures(key, reps, flushed_reps)), flush=True)


# ----------------------------------------------------------------------------- chunked prefill
def prefill_flops(prefix_lens, chunk_lens, H, D) -> int:
    """Causal attention FLOPs: query at position p does 2*D*(p+1) for Q K^T and the
    same for P V, per head."""
    total = 0
    for L0, n in zip(prefix_lens, chunk_lens):
        # sum over positions L0 .. L0+n-1 of (p + 1)
        total += n * (2 * L0 + n + 1) // 2
    return 4 * D * H * total


def prefill_figures(reps=20, flushed_reps=50, e2e=True, device_rows=False, sample_clocks=False, dtype="f16"):
    """pa_prefill on the chunked-prefill batch (16 sequences, prefix ~U[0, 3072], a
    512-token chunk each, H=32, D=128, B=16, fp16): TFLOP/s of causal FLOPs, mean of
    ``reps`` back-to-back launches queued behind a GPU sleep (the batch's K/V, ~0.9 GB,
    exceeds L2), and the median of ``flushed_reps`` launches each timed alone after a
    read of twice the L2 size.  ``e2e``: the chunk step through host buffers (q, k, v
    rows in from pinned memory, pa_cache_append, pa_prefill, output back)."""
    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa
    import workloads

    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    w = workloads.prefill_batch(dtype=dtype)
    eng = pa.PagedKVEngine(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype, free_order=w.free_order,
                           device=dev, max_seqs=64,
                           max_blocks_per_seq=max(-(-L // w.block_size) for L in w.final_lens.values()))
    (op,) = w.prefill_ops
    if device_rows:
        replay_device_rows(eng, w, 5000 + w.seed)
    else:
        for i, o in enumerate(w.ops[:op]):
            if o[0] == "add":
                eng.add_seq(o[1], *w.rows(i))
            elif o[0] == "extend":
                eng.extend(o[1], *w.rows(i))
    seqs, counts = w.ops[op][1], w.ops[op][2]
    tables, lens = eng.bm.block_tables(seqs, eng.max_blocks)
    qs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    tt, ll, qq = (torch.from_numpy(x).to(dev) for x in (tables, lens, qs))
    if device_rows:
        g = torch.Generator(device=dev)
        g.manual_seed(6000 + w.seed)
        q = torch.randn(int(qs[-1]), w.num_heads, w.head_dim, generator=g, device=dev).to(
            pa.engine.TORCH_DTYPES[w.dtype])
    else:
        q = pa.to_device_rows(w.query(op), w.dtype, dev)
    out = torch.empty_like(q)

    def launch():
        pa.pa_prefill(q, eng.k_cache, eng.v_cache, tt, ll, qq, w.scale, out)

    clocks = ClockSampler(dev.index, interval_ms=20) if sample_clocks else None
    if clocks:
        clocks.start()
    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(2_000_000)
    e0.record(st)
    for _ in range(reps):
        launch()
    e1.record(st)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    # the same launch timed alone after a read of twice the L2 size
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 132 * 2 ** 20
    flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(flushed_reps)]
    for a, b in ev:
        flush.sum()
        a.record(st)
        launch()
        b.record(st)
    torch.cuda.synchronize()
    us_flushed = float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e3
    clk = clocks.stop() if clocks else None
    del flush
    prefix = [int(L) - int(n) for L, n in zip(lens, counts)]
    flops = prefill_flops(prefix, counts, w.num_heads, w.head_dim)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        peak, src = 1900.0, "fallback (1.9 PFLOP/s)"
    tf = flops / (us * 1e-6) / 1e12
    res = {"metric": "chunked prefill attention TFLOP/s (causal FLOPs)", "workload": w.name,
           "prefill_us": round(us, 2), "flops": flops, "tflops": round(tf, 1),
           "timing": f"mean of {reps} back-to-back launches queued behind a GPU sleep",
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tf / peak, 4), "peak_source": src},
           "flushed": {"prefill_us_median": round(us_flushed, 2), "launches": flushed_reps,
                       "tflops": round(flops / (us_flushed * 1e-6) / 1e12, 1)},
           "query_rows": int(qs[-1]), "dtype": w.dtype,
           "data": "device-drawn rows (timing only)" if device_rows else "host-drawn rows (the workload generator)"}
    if clk is not None:
        res["clocks"] = clk
    if e2e:
        # End to end through host buffers: every step copies the chunk's queries and its
        # new K/V rows from pinned host memory, appends the rows at their slots (the
        # values already there: the cache is unchanged), prefills, and copies the output
        # back.  The copies are pipelined over two buffer sets: step k+1's inputs travel on
        # one copy stream and step k-1's output on another while step k computes.
        slot_list = []
        for s_, L_, n_ in zip(seqs, lens, counts):
            slot_list += [eng.bm.slot(s_, p_) for p_ in range(int(L_) - int(n_), int(L_))]
        slots = torch.tensor(slot_list, dtype=torch.int32, device=dev)
        kn = eng.k_cache.view(-1, w.num_heads, w.head_dim)[slots.long()]
        vn = eng.v_cache.view(-1, w.num_heads, w.head_dim)[slots.long()]
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, kn, vn))
        hout = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
        bufs = [(torch.empty_like(q), torch.empty_like(kn), torch.empty_like(vn), torch.empty_like(out))
                for _ in range(2)]
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_read = [torch.cuda.Event() for _ in range(2)]
        k_e2e = 10

        def load(k):
            dq, dk, dv, _ = bufs[k % 2]
            with torch.cuda.stream(cin):
                if k >= 2:
                    cin.wait_event(ev_done[k % 2])
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ev_in[k % 2].record(cin)

        def run(n):
            load(0)
            for k in range(n):
                b_ = k % 2
                dq, dk, dv, do = bufs[b_]
                if k + 1 < n:
                    load(k + 1)
                st.wait_event(ev_in[b_])
                if k >= 2:
                    st.wait_event(ev_read[b_])
                pa.pa_cache_append(dk, dv, slots, eng.k_cache, eng.v_cache)
                pa.pa_prefill(dq, eng.k_cache, eng.v_cache, tt, ll, qq, w.scale, do)
                ev_done[b_].record(st)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_done[b_])
                    hout[b_].copy_(do, non_blocking=True)
                    ev_read[b_].record(cout)
            st.wait_stream(cin)
            st.wait_stream(cout)

        run(3)
        torch.cuda.synchronize()
        e0.record(st)
        cin.wait_event(e0)
        run(k_e2e)
        e1.record(st)
        torch.cuda.synchronize()
        e2e_us = e0.elapsed_time(e1) / k_e2e * 1e3
        for h_ in hout:
            assert torch.equal(h_.view(torch.int16), out.cpu().view(torch.int16))
        hout = hout[0]
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h = hout.numel() * hout.element_size()
        res["e2e"] = {"us_per_step": round(e2e_us, 2), "tflops": round(flops / (e2e_us * 1e-6) / 1e12, 1),
                      "steps": k_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "step": "queries and the chunk's K/V rows copied from pinned host memory, "
                              "pa_cache_append of the chunk, pa_prefill, output copied back; copies "
                              "pipelined over two buffer sets on two copy streams"}
    del eng
    torch.cuda.empty_cache()
    return res


def prefill_bench(reps=20, dtype="f16"):
    """pa_prefill on the chunked-prefill batch; one JSON line (TFLOP/s)."""
    import torch

    torch.cuda.set_device(0)
    print(json.dumps(prefill_figures(reps, dtype=dtype)), flush=True)


def bench_extras(device, reps=10, flushed_reps=10):
    """The other serving shapes, each on the decode kernel path the engine picks, with
    device-drawn rows: long context 4 x 16384 (split contexts + merge), parallel
    sampling with copy-on-write (plain and through the shared-prefix decode), the
    256-sequence serving mix (with its append), and the chunked prefill.  Then the
    beam-search step loop over forked sequences (plain and shared-prefix decode),
    prompt admission with and without prefix caching, the two cache layouts, and
    decode / prefill throughput against the block size."""
    peak, src = _peaks()
    out = {}

    def decode_entry(key):
        f = decode_figures(key, reps, flushed_reps, device_rows=True, memset=False, append=(key == "4"),
                           sample_clocks=True)
        fl = f["flushed"]
        ent = {"workload": f["name"], "params": f["params"], "seqs": f["seqs"], "sum_len": f["sum_len"],
               "gbps": fl["gbps"], "frac": round(fl["gbps"] / peak, 4), "peak": peak, "peak_source": src,
               "decode_us": fl["decode_us_median"],
               "timing": f"median of {flushed_reps} launches, each timed alone with CUDA events after a read "
                         f"of twice the L2 size",
               "back_to_back": {"decode_us": f["decode_us"], "gbps": f["gbps"], "launches": reps},
               "algorithmic_bytes": f["algorithmic_bytes"], "seqs_per_sec": fl["seqs_per_sec"],
               "clocks": f.get("clocks"), "data": f["data"]}
        if key in ("3", "3s"):
            ent["unique_frame_bytes"] = f["unique_frame_bytes"]
            ent["gbps_unique_frames"] = fl["gbps_unique_frames"]
            ent["frac_unique_frames"] = fl["frac_unique_frames"]
            ent["gbps_logical"] = fl["gbps"]
            ent["cow_copies"] = f["cow_copies"]
        if "append" in f:
            ent["append"] = f["append"]
        return ent

    for key, name in (("2", "cfg2"), ("3", "cfg3"), ("3s", "cfg3_shared"), ("4", "cfg4")):
        out[name] = _guarded(lambda k=key: decode_entry(k))
    out["prefill"] = _guarded(lambda: prefill_figures(reps, flushed_reps, e2e=False, device_rows=True,
                                                      sample_clocks=True))
    # the remaining next-step workloads, compact; every entry is guarded, so that a
    # failure leaves its error in the line instead of losing the line
    out["fork_trees"] = {"pa_decode": _guarded(lambda: fork_tree_bench(emit=False)),
                         "shared_prefix": _guarded(lambda: fork_tree_bench(share=True, emit=False))}
    out["prefix_caching"] = _guarded(lambda: prefix_bench(emit=False))
    out["split_layout"] = _guarded(lambda: split_layout_bench(emit=False))
    out["block_sweep"] = _guarded(lambda: block_sweep(blocks=(8, 16, 32, 64), emit=False))
    return out


# ----------------------------------------------------------------------------- reference arm
def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    budget_steps = args.steps + args.warmup
    res = cpu_baseline_worker(args.config, 0, per_step=True, steps=budget_steps)
    times, byts = res["times"][args.warmup:], res["bytes"][args.warmup:]
    total_t = sum(times)
    value = sum(byts) / total_t / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1000 * total_t / max(1, len(times)), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, same generator as the GPU arm)",
        "config": {"workload": "decode batch: 64 seqs, context ~U[512,2048], 32 heads, head_dim 128, "
                               "block_size 16, fp16 storage",
                   "step": "one sequence of the batch per step (bounded sample)"},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": res["sample"], "value": round(value, 4),
                         "unit": UNIT},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefix_bench(n_requests=16, system_len=2048, user_len=512, reps=10, emit=True):
    """Admission of requests that share a system prompt: host block manager, cache
    append of the rows that must be computed, causal prefill of those tokens.
    Three ways: no prefix cache (every prompt in full), prefix cache starting empty
    (the first request computes the system prompt), prefix cache already holding it.
    One JSON line per run: prompt tokens admitted per second on the GPU (the append
    of the computed rows + the prefill, CUDA events) and end to end (host block
    manager + launches + GPU, one synchronize per admission; the block manager is
    reset to its starting state before each timed admission, outside the timing),
    with the parts."""
    import time

    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    H, D, B, dtype = 32, 128, 16, "f16"
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([2024, 0])))
    system = rng.integers(0, 1 << 20, size=system_len).astype(np.int32)
    prompts = [np.concatenate([system, rng.integers(0, 1 << 20, size=user_len).astype(np.int32)])
               for _ in range(n_requests)]
    warm_prompt = np.concatenate([system, np.zeros(1, np.int32)])
    L = system_len + user_len
    nb = int(1.2 * n_requests * -(-L // B)) + 8
    eng = pa.PagedKVEngine(nb, B, H, D, dtype, device=dev, max_seqs=max(64, n_requests), max_blocks_per_seq=-(-L // B))
    g = torch.Generator(device=dev).manual_seed(7)
    k_rows = torch.randn((n_requests, L, H, D), generator=g, device=dev, dtype=torch.float32).to(torch.float16)
    v_rows = torch.randn((n_requests, L, H, D), generator=g, device=dev, dtype=torch.float32).to(torch.float16)
    q_rows = torch.randn((n_requests * L, H, D), generator=g, device=dev, dtype=torch.float32).to(torch.float16)
    scale = 1.0 / float(np.sqrt(D))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def reset(mode):
        """A fresh block manager (not timed): empty, or holding the system prompt."""
        eng.bm = pa.BlockManager(nb, B)
        if mode == "warm":  # an earlier request left the system prompt in the cache
            eng.bm.add_seq_cached(10 ** 6, warm_prompt)
            eng.bm.free(10 ** 6)

    def host_admit(mode):
        """Block manager only: per request (n_cached, slots of the rows to write)."""
        res = []
        for i, toks in enumerate(prompts):
            if mode == "none":
                res.append((0, eng.bm.add_seq(i, L)))
            else:
                res.append(eng.bm.add_seq_cached(i, toks))
        return res

    out = {}
    for mode in ("none", "cold", "warm"):
        # the rows a model would produce for the tokens that must be computed, laid
        # out contiguously per admission (built once, outside the timed region)
        reset(mode)
        res = host_admit(mode)
        counts = [L - n for n, _ in res]
        krows = torch.cat([k_rows[i, n:] for i, (n, _) in enumerate(res)])
        vrows = torch.cat([v_rows[i, n:] for i, (n, _) in enumerate(res)])
        q = torch.cat([q_rows[i * L + n:(i + 1) * L] for i, (n, _) in enumerate(res)])
        flops = sum(prefill_flops([n], [L - n], H, D) for n, _ in res)
        seqs = list(range(n_requests))

        def admit():
            t = time.perf_counter()
            r = host_admit(mode)
            t_bm = time.perf_counter() - t
            ev[0].record(st)
            eng.write_rows(np.concatenate([sl for _, sl in r]), krows, vrows)
            ev[1].record(st)
            eng.prefill(seqs, counts, q, scale)
            ev[2].record(st)
            torch.cuda.synchronize()
            return t_bm, ev[0].elapsed_time(ev[1]) / 1e3, ev[1].elapsed_time(ev[2]) / 1e3

        for _ in range(3):
            reset(mode)
            admit()
        walls, app, pf, bm_t = [], [], [], []
        for _ in range(reps):
            reset(mode)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            t_bm, t_ap, t_pf = admit()
            walls.append(time.perf_counter() - t0)
            app.append(t_ap)
            pf.append(t_pf)
            bm_t.append(t_bm)
        med = lambda x: float(np.median(x))
        wall, ap, pfm, tb = med(walls), med(app), med(pf), med(bm_t)
        out[mode] = {"ms_e2e": round(wall * 1e3, 3), "prompt_tokens_per_s_e2e": round(n_requests * L / wall),
                     "gpu_ms": round((ap + pfm) * 1e3, 3),
                     "prompt_tokens_per_s_gpu": round(n_requests * L / (ap + pfm)),
                     "tokens_computed": sum(counts), "tokens_from_cache": n_requests * L - sum(counts),
                     "append_ms": round(ap * 1e3, 3), "prefill_ms": round(pfm * 1e3, 3),
                     "prefill_tflops": round(flops / pfm / 1e12, 1), "host_block_manager_ms": round(tb * 1e3, 3)}
    line = {"metric": "prompt admission tokens/s with prefix caching (host block manager + append + prefill)",
            "workload": f"{n_requests} requests x (system {system_len} + user {user_len}), H={H}, D={D}, B={B}, "
                        f"{dtype}", "reps": reps, "statistic": "median", **out,
            "speedup_gpu_warm_vs_none": round(out["none"]["gpu_ms"] / out["warm"]["gpu_ms"], 2),
            "speedup_gpu_cold_vs_none": round(out["none"]["gpu_ms"] / out["cold"]["gpu_ms"], 2),
            "speedup_e2e_warm_vs_none": round(out["none"]["ms_e2e"] / out["warm"]["ms_e2e"], 2),
            "speedup_e2e_cold_vs_none": round(out["none"]["ms_e2e"] / out["cold"]["ms_e2e"], 2)}
    del eng, k_rows, v_rows, q_rows
    torch.cuda.empty_cache()
    if emit:
        print(json.dumps(line), flush=True)
    return line


def fork_tree_bench(n_prompts=8, prompt_len=2048, width=8, steps=64, share=False, emit=True):
    """Beam search over forked sequences, the whole step loop on one GPU: host block
    manager (step with copy-on-write, then the selection's forks and frees in one
    batched call each), staged
    upload, pa_copy_blocks, pa_cache_append and pa_decode over every live beam.
    One JSON line: step time end to end, decode time (CUDA events around a repeat of
    each step's decode queued behind a short GPU sleep, so host enqueue gaps are not
    counted), decode GB/s of logical bytes (what the beams attend) and of the unique
    frames they hold."""
    import time

    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    H, D, B, dtype = 32, 128, 16, "f16"
    w = workloads.beam_search(n_prompts, prompt_len, width, steps, H=H, D=D, B=B, dtype=dtype, seed=77)
    nbeams = n_prompts * width
    mb = -(-(prompt_len + steps) // B)
    g = torch.Generator(device=dev).manual_seed(9)
    prompt_k = torch.randn((prompt_len, H, D), generator=g, device=dev).to(torch.float16)
    prompt_v = torch.randn((prompt_len, H, D), generator=g, device=dev).to(torch.float16)
    step_k = torch.randn((nbeams, H, D), generator=g, device=dev).to(torch.float16)
    step_v = torch.randn((nbeams, H, D), generator=g, device=dev).to(torch.float16)
    q = torch.randn((nbeams, H, D), generator=g, device=dev).to(torch.float16)
    out = torch.empty_like(q)
    out2 = torch.empty_like(q)
    scale = 1.0 / float(np.sqrt(D))
    row = 2 * H * D * 2  # K + V bytes of one token of one sequence

    def run(record):
        eng = pa.PagedKVEngine(w.num_blocks, B, H, D, dtype, free_order=w.free_order, device=dev,
                               max_seqs=nbeams, max_blocks_per_seq=mb)
        ops = w.ops
        stats = []
        t_first = None  # the timed loop starts at the first step (after the prompts are written)
        i = 0
        while i < len(ops):
            op = ops[i]
            if op[0] == "step" and t_first is None:
                torch.cuda.synchronize()
                t_first = time.perf_counter()
            if op[0] == "add":
                eng.add_seq(op[1], prompt_k, prompt_v)
            elif op[0] in ("fork", "free"):
                # one selection (every fork and free up to the next step) in two calls: the
                # forks in order, then the frees in order (same state as the interleaved
                # order: tests/test_fork_trees_host.py)
                j = i
                while j < len(ops) and ops[j][0] in ("fork", "free"):
                    j += 1
                forks = [o for o in ops[i:j] if o[0] == "fork"]
                frees = [o[1] for o in ops[i:j] if o[0] == "free"]
                if forks:
                    eng.fork_many([o[1] for o in forks], [o[2] for o in forks])
                if frees:
                    eng.free_many(frees)
                i = j
                continue
            elif op[0] == "step":
                live = op[1]
                assert ops[i + 1][0] == "attend" and ops[i + 1][1] == live
                prm = {"share_prefix": 1} if share else {}
                _, nc, lens = eng.decode_step(live, step_k, step_v, q, scale, out=out, params=prm)
                if record:
                    # decode time: the same decode again behind a short GPU sleep, so the host
                    # has enqueued it before the start event runs and the events bracket GPU
                    # work only (the host side of a step takes longer than a shared decode)
                    e = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                    torch.cuda._sleep(400_000)
                    eng.attend(live, q, scale, out=out2, params=prm, events=e)
                    tables, ln = eng.bm.block_tables(live, mb)
                    unique = len(set(tables[tables >= 0].tolist()))
                    stats.append((e, int(ln.sum()) * row, unique * B * row, nc))
                else:
                    stats.append((None, 0, 0, nc))
                i += 1
            i += 1
        torch.cuda.synchronize()
        return stats, time.perf_counter() - t_first

    run(False)
    steps_done, total = run(False)
    n_steps = len(steps_done)
    stats, _ = run(True)  # decode events and byte counts (host bookkeeping kept out of the timed run)
    dec = np.array([e[0].elapsed_time(e[1]) / 1e3 for e, *_ in stats])
    logical = np.array([x[1] for x in stats], np.float64)
    unique = np.array([x[2] for x in stats], np.float64)
    copies = int(sum(x[3] for x in stats))
    res = {
        "metric": "beam-search decode step over forked sequences (block manager + copy-on-write + append + decode)",
        "workload": w.name, "share_prefix": int(share), "beams": nbeams, "steps": len(stats),
        "ms_per_step_e2e": round(total / n_steps * 1e3, 3),
        "e2e_region": "from the first step to the last (block manager, forks/frees, uploads, copies, append, decode)",
        "decode_us_median": round(float(np.median(dec)) * 1e6, 2),
        "decode_gbs_logical": round(float(np.sum(logical) / np.sum(dec)) / 1e9, 1),
        "decode_gbs_unique_frames": round(float(np.sum(unique) / np.sum(dec)) / 1e9, 1),
        "logical_over_unique_bytes": round(float(np.sum(logical) / np.sum(unique)), 2),
        "cow_copies": copies, "cow_copies_per_step": round(copies / len(stats), 2)}
    torch.cuda.empty_cache()
    if emit:
        print(json.dumps(res), flush=True)
    return res


def block_sweep(blocks=(8, 16, 32, 64, 128, 256), reps=20, emit=True):
    """Block size B against throughput, one JSON line per B: pa_decode on the decode
    batch's lengths (64 sequences, L ~ U[512, 2048], H=32, D=128, fp16; GB/s of
    algorithmic bytes) and pa_prefill on the chunked-prefill batch's shapes (16 x
    512-token chunks after prefixes ~U[0, 3072]; TFLOP/s of causal FLOPs; B <= 128).
    Caches are filled on the device; frames come from a shuffled free list."""
    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    H, D = 32, 128
    dec_lens = [w_L for w_L in workloads.build(1).final_lens.values()]
    pw = workloads.prefill_batch()
    (pop,) = pw.prefill_ops
    pre_lens = [pw.final_lens[s] - n for s, n in zip(pw.ops[pop][1], pw.ops[pop][2])]
    chunks = list(pw.ops[pop][2])
    g = torch.Generator(device=dev).manual_seed(11)

    def engine(lengths, B):
        need = sum(-(-L // B) for L in lengths)
        nb = int(1.2 * need) + 1
        order = np.random.Generator(np.random.PCG64(B)).permutation(nb).astype(np.int32)
        eng = pa.PagedKVEngine(nb, B, H, D, "f16", free_order=order, device=dev, max_seqs=len(lengths),
                               max_blocks_per_seq=max(-(-L // B) for L in lengths))
        for s, L in enumerate(lengths):
            eng.bm.add_seq(s, L)
        eng.k_cache.normal_(generator=g)
        eng.v_cache.normal_(generator=g)
        return eng

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    lines = []
    for B in blocks:
        line = {"metric": "block size sweep", "B": B}
        eng = engine(dec_lens, B)
        S = len(dec_lens)
        ids = list(range(S))
        tables, lens = eng.bm.block_tables(ids, eng.max_blocks)
        td, ld = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
        q = torch.randn((S, H, D), generator=g, device=dev).to(torch.float16)
        out = torch.empty_like(q)
        try:
            t = timed(lambda: pa.pa_decode(q, eng.k_cache, eng.v_cache, td, ld, 0.0883883, out))
        except pa.PAError as e:
            line["decode"] = f"unsupported: {e}"
        else:
            byts = sum(2 * L * H * D * 2 + 4 * -(-L // B) for L in dec_lens) + 4 * S + 2 * S * H * D * 2
            line.update({"decode_us": round(t * 1e6, 2), "decode_gbs": round(byts / t / 1e9, 1)})
        del eng
        if B <= 128:
            eng = engine([a + b for a, b in zip(pre_lens, chunks)], B)
            S = len(chunks)
            ids = list(range(S))
            tables, lens = eng.bm.block_tables(ids, eng.max_blocks)
            qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
            td, ld, qd = (torch.from_numpy(x).to(dev) for x in (tables, lens, qs))
            qq = torch.randn((int(qs[-1]), H, D), generator=g, device=dev).to(torch.float16)
            oo = torch.empty_like(qq)
            t = timed(lambda: pa.pa_prefill(qq, eng.k_cache, eng.v_cache, td, ld, qd, 0.0883883, oo))
            fl = prefill_flops(pre_lens, chunks, H, D)
            line.update({"prefill_us": round(t * 1e6, 2), "prefill_tflops": round(fl / t / 1e12, 1)})
            del eng
        torch.cuda.empty_cache()
        lines.append(line)
        if emit:
            print(json.dumps(line), flush=True)
    return lines


def split_layout_bench(reps=20, emit=True):
    """The two cache layouts head to head, one JSON line per (workload, B): pa_decode
    on [num_blocks, B, H, D] caches and pa_decode_split on the layout of the pages'
    kernel signature (k [num_blocks, H, D/x, B, x], v [num_blocks, H, D, B]); same
    lengths, same frames, caches filled on the device; GB/s of algorithmic bytes."""
    import numpy as np
    import torch

    import paged_kv_cache_126_gb300 as pa
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    H, D = 32, 128
    g = torch.Generator(device=dev).manual_seed(13)
    cases = [("decode batch: 64 seqs, L~U[512,2048]", list(workloads.build(1).final_lens.values())),
             ("long context: 4 x 16384", [16384] * 4)]

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    lines = []
    for name, lens in cases:
        for B in (8, 16, 32):
            S = len(lens)
            need = sum(-(-L // B) for L in lens)
            nb = int(1.2 * need) + 1
            order = np.random.Generator(np.random.PCG64(B)).permutation(nb).astype(np.int32)
            bm = pa.BlockManager(nb, B, order)
            for s, L in enumerate(lens):
                bm.add_seq(s, L)
            mb = max(-(-L // B) for L in lens)
            tables, ln = bm.block_tables(list(range(S)), mb)
            td, ld = torch.from_numpy(tables).to(dev), torch.from_numpy(ln).to(dev)
            q = torch.randn((S, H, D), generator=g, device=dev).to(torch.float16)
            out = torch.empty_like(q)
            byts = sum(2 * L * H * D * 2 + 4 * -(-L // B) for L in lens) + 4 * S + 2 * S * H * D * 2
            line = {"metric": "cache layout: row [nb,B,H,D] vs split [nb,H,D/x,B,x]/[nb,H,D,B] decode",
                    "workload": name, "B": B}
            kc = torch.empty((nb, B, H, D), dtype=torch.float16, device=dev).normal_(generator=g)
            vc = torch.empty((nb, B, H, D), dtype=torch.float16, device=dev).normal_(generator=g)
            t = timed(lambda: pa.pa_decode(q, kc, vc, td, ld, 0.0883883, out))
            line["row_gbs"] = round(byts / t / 1e9, 1)
            del kc, vc
            ks = torch.empty((nb, H, D // 8, B * 8), dtype=torch.float16, device=dev).normal_(generator=g)
            vs = torch.empty((nb, H, D, B), dtype=torch.float16, device=dev).normal_(generator=g)
            t = timed(lambda: pa.pa_decode_split(q, ks, vs, td, ld, 0.0883883, out))
            line["split_gbs"] = round(byts / t / 1e9, 1)
            del ks, vs
            torch.cuda.empty_cache()
            lines.append(line)
            if emit:
                print(json.dumps(line), flush=True)
    return lines


def _bm_replay(pa, w):
    """Run a workload's block-manager ops through libpa's native manager (host only)."""
    bm = pa.BlockManager(w.num_blocks, w.block_size, w.free_order)
    for op in w.ops:
        kind = op[0]
        if kind == "add":
            bm.add_seq(op[1], op[2])
        elif kind == "fork":
            bm.fork(op[1], op[2])
        elif kind == "step":
            bm.step(op[1])
        elif kind == "extend":
            bm.extend(op[1], op[2])
        elif kind == "free":
            bm.free(op[1])
        elif kind == "add_tokens":
            bm.add_seq_cached(op[1], op[2])
        elif kind == "extend_tokens":
            bm.extend_tokens(op[1], op[2])
        elif kind == "step_tokens":
            bm.step_tokens(op[1], op[2])
    return bm


def memory_report(l_max=8192):
    """Memory held by the paged cache at each workload's final state (host only).

    Paged: frames in use x B slots against the token slots they hold (waste is
    confined to each sequence's last frame, under B slots); frames shared by forked
    sequences are held once.  Contiguous counterfactual: every live sequence reserves
    max(l_max, its workload's longest sequence) slots.
    """
    import workloads
    import paged_kv_cache_126_gb300 as pa

    cases = [(str(k), workloads.build(k)) for k in (0, 1, "1x", 2, 3, 4)]
    cases.append(("beam", workloads.beam_search(8, 2048, 8, 64, H=32, D=128, B=16, dtype="f16", seed=31)))
    cases.append(("prefix", workloads.shared_prefix(16, 2048, [512] * 16, H=32, D=128, B=16, dtype="f16",
                                                    seed=21)))
    for key, w in cases:
        t0 = time.perf_counter()
        bm = _bm_replay(pa, w)
        u = bm.usage()
        host_ms = (time.perf_counter() - t0) * 1e3
        B = w.block_size
        row_bytes = 2 * w.num_heads * w.head_dim * w.elem_bytes  # K and V of one token
        slots = u["frames_in_use"] * B
        lmax = max([l_max] + [int(x) for x in w.final_lens.values()])
        reserve = u["num_seqs"] * lmax
        print(json.dumps({
            "memory": w.name, "key": key, "block_size": B, "seqs": u["num_seqs"],
            "frames_in_use": u["frames_in_use"], "frames_total": u["frames_total"],
            "frames_cached": u["frames_cached"], "slots_allocated": slots, "slots_filled": u["slots_filled"],
            "tokens_logical": u["tokens_logical"], "table_entries": u["table_entries"],
            "paged_waste_pct": round(100.0 * (1 - u["slots_filled"] / slots), 3) if slots else 0.0,
            "max_seq_waste_slots": u["max_seq_waste"], "waste_bound_slots": B - 1,
            "shared_frames_saving_pct": (round(100.0 * (1 - u["frames_in_use"] / u["table_entries"]), 2)
                                         if u["table_entries"] else 0.0),
            "contiguous_l_max": lmax,
            "contiguous_waste_pct": round(100.0 * (1 - u["tokens_logical"] / reserve), 2) if reserve else 0.0,
            "kv_gb_paged": round(slots * row_bytes / 1e9, 4),
            "kv_gb_contiguous": round(reserve * row_bytes / 1e9, 4),
            "replay_host_ms": round(host_ms, 1)}), flush=True)
        bm.close()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1600)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batches", type=int, default=16, help="resident copies of the batch decoded in rotation")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-budget", type=float, default=None,
                    help="seconds of oracle decode time per CPU measurement (8: one thread, then each of the all-cores workers)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--config", default="1")
    ap.add_argument("--cpu-worker", default=None)
    ap.add_argument("--prefill", action="store_true", help="time pa_prefill on the chunked-prefill batch instead")
    ap.add_argument("--prefill-dtype", choices=["f16", "bf16"], default="f16")
    ap.add_argument("--prefix", action="store_true", help="time prompt admission with and without prefix caching")
    ap.add_argument("--fork-trees", action="store_true", help="time the beam-search step loop over forked sequences")
    ap.add_argument("--block-sweep", action="store_true", help="decode and prefill throughput against block size")
    ap.add_argument("--split-layout", action="store_true", help="decode throughput of the two cache layouts")
    ap.add_argument("--sweep", default=None, metavar="KEYS",
                    help="time pa_decode on each listed workload instead (comma list of 0,1,1x,2,2n,3,3c,3s,4,4d "
                         "or 'all'; 4d = the serving mix's first 48 sequences)")
    ap.add_argument("--cpu-seed-shift", type=int, default=0)
    ap.add_argument("--cpu-sweep", action="store_true",
                    help="time the oracle's decode on the host per workload, one thread and all affine cores")
    ap.add_argument("--memory", action="store_true",
                    help="memory held by the paged cache vs a contiguous reservation, per workload (host only)")
    args = ap.parse_args()
    if args.memory:
        memory_report()
        return
    if args.cpu_sweep:
        cpu_sweep(budget_s=args.cpu_budget or 8.0)
        return
    if args.prefix:
        prefix_bench()
        return
    if args.fork_trees:
        fork_tree_bench()
        fork_tree_bench(share=True)
        return
    if args.block_sweep:
        block_sweep()
        return
    if args.split_layout:
        split_layout_bench()
        return
    if args.prefill:
        prefill_bench(dtype=args.prefill_dtype)
        return
    if args.sweep is not None:
        keys = SWEEP_KEYS if args.sweep == "all" else tuple(args.sweep.split(","))
        sweep(keys)
        return
    if args.config not in ("1", "1x"):
        raise SystemExit("the bench times the decode batch workload (1) or its fixed 64x2048 form (1x)")
    args.config = 1 if args.config == "1" else "1x"
    if args.cpu_worker is not None:
        cfg = args.cpu_worker if args.cpu_worker == "1x" else int(args.cpu_worker)
        print(json.dumps(cpu_baseline_worker(cfg, args.cpu_budget or 12.0, seed_shift=args.cpu_seed_shift)), flush=True)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
