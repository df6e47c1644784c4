"""Replay a workload through the oracle block manager, cache model and attention.

Issue order inside a decode step: the step's copy-on-write frame copies are
applied before the step's new rows are written (a copy reads the shared frame as
it was before any writer of this step touched it).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .attention import paged_decode, paged_prefill
from .block_manager import OracleBlockManager
from .cache import OracleKVCache
from .prefix_cache import OraclePrefixBlockManager

TOKEN_OPS = ("add_tokens", "extend_tokens", "step_tokens", "prefill_new")


@dataclass
class ReplayResult:
    bm: OracleBlockManager
    cache: OracleKVCache | None
    # per op index: {"slots": [...], "copies": [(src, dst), ...]} for add/step ops
    trace: dict = field(default_factory=dict)
    # per op index: BM snapshot after the op
    snapshots: dict = field(default_factory=dict)
    # per attend op index: float64 [n, H, D] (rows of sequences not kept are NaN)
    outputs: dict = field(default_factory=dict)
    # per attend op index: (tables, lens) the attention used, in the op's seq order
    attend_meta: dict = field(default_factory=dict)
    # per token-driven sequence: tokens its admission found in the cache
    n_cached: dict = field(default_factory=dict)


def _kept_frames(w, keep_seqs):
    """Frames whose contents reach the kept sequences: the frames their tables name
    when they attend (and at the end), plus every frame a copy-on-write copy into one
    of those read from, transitively.  Only the index-driven ops occur here: replay()
    refuses ``keep_seqs`` for token-driven workloads."""
    bm = OracleBlockManager(w.num_blocks, w.block_size, w.free_order)
    edges = []
    seen = set()
    for op in w.ops:
        kind = op[0]
        if kind == "add":
            bm.add_seq(op[1], op[2])
        elif kind == "fork":
            bm.fork(op[1], op[2])
        elif kind == "step":
            _, copies = bm.step(op[1])
            edges.extend(copies)
        elif kind == "extend":
            _, copies = bm.extend(op[1], op[2])
            edges.extend(copies)
        elif kind == "free":
            bm.free(op[1])
        elif kind in ("prefill", "attend"):
            for s in op[1]:
                if s in keep_seqs:
                    seen.update(bm.tables[s])
        else:
            raise ValueError(f"op {op[0]!r} cannot be replayed for a subset of sequences")
    for s in keep_seqs:
        if s in bm.tables:
            seen.update(bm.tables[s])
    changed = True
    while changed:
        changed = False
        for src, dst in edges:
            if dst in seen and src not in seen:
                seen.add(src)
                changed = True
    return seen


def replay(w, keep_seqs=None, with_cache: bool = True, snapshots: bool = False) -> ReplayResult:
    """Run every op of ``w``; attention only for ``keep_seqs`` (all if None)."""
    keep = None if keep_seqs is None else set(int(s) for s in keep_seqs)
    tokens = any(op[0] in TOKEN_OPS for op in w.ops)
    if tokens and keep is not None:
        raise ValueError("token-driven workloads replay every sequence")
    frames = None if keep is None else _kept_frames(w, keep)
    bm = (OraclePrefixBlockManager if tokens else OracleBlockManager)(w.num_blocks, w.block_size, w.free_order)
    cache = (OracleKVCache(w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.dtype, keep=frames)
             if with_cache else None)
    res = ReplayResult(bm=bm, cache=cache)
    B = w.block_size
    for i, op in enumerate(w.ops):
        kind = op[0]
        if kind == "add":
            slots = bm.add_seq(op[1], op[2])
            res.trace[i] = {"slots": slots, "copies": []}
            if cache is not None and slots and (frames is None or any(s // B in frames for s in slots)):
                k, v = w.rows(i)
                cache.write(slots, k, v)
        elif kind == "fork":
            bm.fork(op[1], op[2])
        elif kind == "step":
            slots, copies = bm.step(op[1])
            res.trace[i] = {"slots": slots, "copies": copies}
            if cache is not None:
                for src, dst in copies:
                    cache.copy_block(src, dst)
                if frames is None or any(s // B in frames for s in slots):
                    k, v = w.rows(i)
                    cache.write(slots, k, v)
        elif kind == "extend":
            slots, copies = bm.extend(op[1], op[2])
            res.trace[i] = {"slots": slots, "copies": copies}
            if cache is not None:
                for src, dst in copies:
                    cache.copy_block(src, dst)
                if frames is None or any(s // B in frames for s in slots):
                    k, v = w.rows(i)
                    cache.write(slots, k, v)
        elif kind == "prefill":
            seqs, counts = op[1], op[2]
            tables = [list(bm.tables[s]) for s in seqs]
            lens = [bm.lens[s] for s in seqs]
            res.attend_meta[i] = (tables, lens)
            if cache is not None:
                q = w.query(i)
                qs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
                out = np.full(q.shape, np.nan)
                for j, s in enumerate(seqs):
                    if keep is None or s in keep:
                        a, b = qs[j], qs[j + 1]
                        out[a:b] = paged_prefill(q[a:b], cache, [tables[j]], [lens[j]], [0, b - a], w.scale)
                res.outputs[i] = out
        elif kind == "add_tokens":
            n_cached, slots = bm.add_seq_cached(op[1], op[2])
            res.n_cached[op[1]] = n_cached
            res.trace[i] = {"slots": slots, "copies": [], "n_cached": n_cached}
            if cache is not None and slots:
                k, v = w.token_rows(i)
                cache.write(slots, k[n_cached:], v[n_cached:])
        elif kind in ("extend_tokens", "step_tokens"):
            if kind == "extend_tokens":
                slots, copies = bm.extend(op[1], len(op[2]), list(op[2]))
            else:
                slots, copies = bm.step(list(op[1]), list(op[2]))
            res.trace[i] = {"slots": slots, "copies": copies}
            if cache is not None:
                for src, dst in copies:
                    cache.copy_block(src, dst)
                k, v = w.token_rows(i)
                cache.write(slots, k, v)
        elif kind == "prefill_new":
            seqs = op[1]
            tables = [list(bm.tables[s]) for s in seqs]
            lens = [bm.lens[s] for s in seqs]
            counts = [lens[j] - res.n_cached[s] for j, s in enumerate(seqs)]
            res.attend_meta[i] = (tables, lens, counts)
            if cache is not None:
                qs = w.position_queries(i)
                outs = []
                for j, s in enumerate(seqs):
                    q = qs[j][lens[j] - counts[j]:lens[j]]
                    outs.append(paged_prefill(q, cache, [tables[j]], [lens[j]], [0, counts[j]], w.scale))
                res.outputs[i] = outs
        elif kind == "free":
            bm.free(op[1])
        elif kind == "attend":
            seqs = op[1]
            tables = [list(bm.tables[s]) for s in seqs]
            lens = [bm.lens[s] for s in seqs]
            res.attend_meta[i] = (tables, lens)
            if cache is not None:
                q = w.query(i)
                out = np.full((len(seqs), w.num_heads, w.head_dim), np.nan)
                idx = [j for j, s in enumerate(seqs) if keep is None or s in keep]
                if idx:
                    out[idx] = paged_decode(q[idx], cache, [tables[j] for j in idx],
                                            [lens[j] for j in idx], w.scale)
                res.outputs[i] = out
        else:
            raise ValueError(f"unknown op {op!r}")
        if snapshots:
            res.snapshots[i] = bm.snapshot()
    return res
