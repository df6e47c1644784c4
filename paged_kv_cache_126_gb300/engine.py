"""PagedKVEngine: one device's paged K/V caches driven by libpa.

The engine owns the two caches [num_blocks, B, H, D] (torch device memory) and a
libpa host block manager.  A decode step (``decode_step``, one pa_step_decode call) is

    host:   pa_bm_step (slots + copy-on-write pairs, in batch order)
            pa_bm_block_tables (tables + context lengths)
            -> one slot of a mapped pinned staging ring
    device: pa_copy_blocks (only if a shared tail was written; the staged block is
            then uploaded first with one async copy)
            pa_cache_append (the step's new K/V rows; without copies it reads its slots
            from the ring and carries the tables to device memory itself)
            pa_decode (split contexts merged inside the kernel)

all on one stream.  Staging slots form a ring guarded by CUDA events so the host can
prepare step k+1 while the device still runs step k.  The separate operations (step,
attend, ...) stage their small int32 arrays through the engine's own pinned ring.
"""

from __future__ import annotations

import numpy as np
import torch

from ._binding import (
    BlockManager,
    pa_cache_append,
    pa_copy_blocks,
    pa_decode,
    pa_prefill,
    pa_step_decode,
)

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_device_rows(rows, dtype: str, device) -> torch.Tensor:
    """[n, H, D] rows -> device tensor; NumPy bf16 arrives as uint16 bit patterns."""
    if isinstance(rows, torch.Tensor):
        return rows.to(device=device, dtype=TORCH_DTYPES[dtype], non_blocking=True)
    a = np.ascontiguousarray(rows)
    t = torch.from_numpy(a)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16) if a.dtype == np.uint16 else t.to(torch.bfloat16)
    else:
        t = t.to(TORCH_DTYPES[dtype])
    return t.to(device)


class PagedKVEngine:
    def __init__(self, num_blocks: int, block_size: int, num_heads: int, head_dim: int, dtype: str = "f16", *,
                 free_order=None, device=None, max_seqs: int = 256, max_blocks_per_seq: int | None = None,
                 ring: int = 4, stream: torch.cuda.Stream | None = None, auto_share: bool = True):
        # auto_share: decode a batch through the shared-prefix path (pa_decode_ex with
        # share_prefix) when two neighbouring sequences of it start on the same frame
        self.auto_share = bool(auto_share)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.num_blocks, self.B, self.H, self.D = int(num_blocks), int(block_size), int(num_heads), int(head_dim)
        self.dtype = dtype
        self.bm = BlockManager(num_blocks, block_size, free_order)
        shape = (self.num_blocks, self.B, self.H, self.D)
        self.k_cache = torch.zeros(shape, dtype=TORCH_DTYPES[dtype], device=self.device)
        self.v_cache = torch.zeros(shape, dtype=TORCH_DTYPES[dtype], device=self.device)
        self.max_blocks = int(max_blocks_per_seq or num_blocks)
        self.max_seqs = int(max_seqs)
        self.stream = stream
        cap = self.max_seqs * (self.max_blocks + 4) + 64
        self._pin = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(ring)]
        self._pin_np = [p.numpy() for p in self._pin]
        self._dev = torch.empty(cap, dtype=torch.int32, device=self.device)
        self._step_lens = [np.empty(self.max_seqs, np.int32) for _ in range(ring)]  # lengths per native step
        self._events = [torch.cuda.Event() for _ in range(ring)]  # the copy that last read each buffer
        self._recorded = [False] * ring
        self._k = 0
        self._ids_key = None
        self._ids = None

    # -- helpers ----------------------------------------------------------------------------
    def _stream(self):
        return self.stream if self.stream is not None else torch.cuda.current_stream(self.device)

    def _ids_for(self, seqs) -> np.ndarray:
        key = tuple(seqs) if not isinstance(seqs, np.ndarray) else None
        if key is not None and key == self._ids_key:
            return self._ids
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        if key is not None:
            self._ids_key, self._ids = key, ids
        return ids

    def _stage(self):
        """Next pinned staging buffer, once the copy that last read it has run."""
        i = self._k % len(self._pin)
        self._k += 1
        if self._recorded[i]:
            self._events[i].synchronize()
        return i

    def _upload(self, i: int, n: int) -> torch.Tensor:
        if self.stream is None:  # the current stream: no stream switch needed
            self._dev[:n].copy_(self._pin[i][:n], non_blocking=True)
            self._events[i].record()
        else:
            with torch.cuda.stream(self.stream):
                self._dev[:n].copy_(self._pin[i][:n], non_blocking=True)
                self._events[i].record(self.stream)
        self._recorded[i] = True
        return self._dev

    # -- sequence operations -------------------------------------------------------------------
    def add_seq(self, seq: int, k_rows, v_rows) -> np.ndarray:
        """New sequence with a prompt; writes its K/V rows. Returns the slots."""
        k = to_device_rows(k_rows, self.dtype, self.device)
        v = to_device_rows(v_rows, self.dtype, self.device)
        slots = self.bm.add_seq(seq, k.shape[0])
        if len(slots):
            sd = torch.from_numpy(slots).to(self.device)
            pa_cache_append(k, v, sd, self.k_cache, self.v_cache, stream=self._stream())
        return slots

    # -- prefix caching ----------------------------------------------------------------------
    def add_seq_cached(self, seq: int, tokens):
        """Admit a prompt by its token ids, reusing cached blocks of an identical prefix.

        Returns (n_cached, slots): the first n_cached tokens are already in the cache;
        the caller computes only the remaining tokens' K/V rows and writes them with
        write_rows(slots, k, v)."""
        return self.bm.add_seq_cached(seq, tokens)

    def _upload_ints(self, *arrays) -> list:
        """Stage int32 host arrays in one pinned buffer, one async copy; returns
        device views in order (large uploads fall back to a plain copy)."""
        sizes = [int(np.size(a)) for a in arrays]
        total = sum(sizes)
        if total > self._pin[0].numel():
            return [torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(self.device) for a in arrays]
        i = self._stage()
        buf = self._pin_np[i]
        off = 0
        for a, n in zip(arrays, sizes):
            buf[off:off + n] = np.ravel(a)
            off += n
        dev = self._upload(i, total)
        views, off = [], 0
        for a, n in zip(arrays, sizes):
            views.append(dev[off:off + n].view(np.shape(a)))
            off += n
        return views

    def write_rows(self, slots, k_rows, v_rows) -> None:
        """K/V rows [T, H, D] into the caches at the given slots (``pa_cache_append``)."""
        if len(slots) == 0:
            return
        k = to_device_rows(k_rows, self.dtype, self.device)
        v = to_device_rows(v_rows, self.dtype, self.device)
        (sd,) = self._upload_ints(np.asarray(slots, dtype=np.int32))
        pa_cache_append(k, v, sd, self.k_cache, self.v_cache, stream=self._stream())

    def _apply(self, slots, copies, k_rows, v_rows) -> None:
        st = self._stream()
        if len(copies):
            pa_copy_blocks(self.k_cache, self.v_cache, torch.from_numpy(np.ascontiguousarray(copies)).to(self.device),
                           stream=st)
        self.write_rows(slots, k_rows, v_rows)

    def extend_tokens(self, seq: int, tokens, k_rows, v_rows):
        """extend() with the token ids, so blocks it fills become reusable."""
        slots, copies = self.bm.extend_tokens(seq, tokens)
        self._apply(slots, copies, k_rows, v_rows)
        return slots, copies

    def step_tokens(self, seqs, tokens, k_rows, v_rows):
        """step() with the token id appended to each sequence."""
        slots, copies = self.bm.step_tokens(seqs, tokens)
        self._apply(slots, copies, k_rows, v_rows)
        return slots, copies

    def fork(self, parent: int, child: int) -> None:
        """Zero-copy fork in the block manager (frames shared, reference counts raised)."""
        self.bm.fork(parent, child)

    def free(self, seq: int) -> int:
        """Release a sequence; returns PA_WARN_DOUBLE_FREE if it was not live."""
        return self.bm.free(seq)

    def fork_many(self, parents, children) -> None:
        """Forks in order, all or nothing (one block-manager call)."""
        self.bm.fork_many(parents, children)

    def free_many(self, seqs) -> int:
        """Frees in order (one block-manager call)."""
        return self.bm.free_many(seqs)

    def step(self, seqs, k_rows, v_rows):
        """Append one token to each of seqs (batch order). Returns (slots, copies)."""
        ids = self._ids_for(seqs)
        n = len(ids)
        i = self._stage()
        buf = self._pin_np[i]
        slots, copies = buf[:n], buf[n:3 * n].reshape(n, 2)
        nc = self.bm.step_into(ids, slots, copies)
        out_slots, out_copies = slots.copy(), copies[:nc].copy()
        dev = self._upload(i, 3 * n)
        st = self._stream()
        if nc:
            pa_copy_blocks(self.k_cache, self.v_cache, dev[n:n + 2 * nc].view(nc, 2), stream=st)
        k = to_device_rows(k_rows, self.dtype, self.device)
        v = to_device_rows(v_rows, self.dtype, self.device)
        pa_cache_append(k, v, dev[:n], self.k_cache, self.v_cache, stream=st)
        return out_slots, out_copies

    def extend(self, seq: int, k_rows, v_rows):
        """A prompt chunk for one sequence: its K/V rows go to the new slots."""
        k = to_device_rows(k_rows, self.dtype, self.device)
        v = to_device_rows(v_rows, self.dtype, self.device)
        slots, copies = self.bm.extend(seq, k.shape[0])
        st = self._stream()
        if len(copies):
            pa_copy_blocks(self.k_cache, self.v_cache, torch.from_numpy(np.ascontiguousarray(copies)).to(self.device),
                           stream=st)
        if len(slots):
            pa_cache_append(k, v, torch.from_numpy(slots).to(self.device), self.k_cache, self.v_cache, stream=st)
        return slots, copies

    def prefill(self, seqs, counts, q, scale: float, out=None) -> torch.Tensor:
        """Causal attention for the last counts[i] positions of seqs[i]; q rows grouped
        by sequence in order."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = len(ids)
        mb = self.max_blocks
        q = to_device_rows(q, self.dtype, self.device)
        if out is None:
            out = torch.empty_like(q)
        tables = np.empty((max(n, 1), mb), np.int32)
        lens = np.empty(max(n, 1), np.int32)
        self.bm.block_tables_into(ids, mb, tables, lens)
        qs = np.zeros(n + 1, np.int32)
        qs[1:] = np.cumsum(np.asarray(counts, np.int64))
        td, ld, qd = self._upload_ints(tables[:n], lens[:n], qs)
        pa_prefill(q, self.k_cache, self.v_cache, td, ld, qd, scale, out, stream=self._stream())
        return out

    def _decode_params(self, tables: np.ndarray, params):
        """Launch options of one decode: the caller's, else the shared-prefix path when two
        neighbouring sequences of the batch start on the same frame (forks of one parent,
        prompts admitted through the prefix cache), else the defaults."""
        if params is not None or not self.auto_share or tables.shape[0] < 2 or tables.shape[1] == 0:
            return params
        first = tables[:, 0]
        if np.any((first[1:] == first[:-1]) & (first[1:] >= 0)):
            return {"share_prefix": 1}
        return None

    def attend(self, seqs, q, scale: float, out=None, params=None, events=None) -> torch.Tensor:
        """Decode attention for seqs with queries q [n, H, D].  ``events`` (start, end):
        CUDA events recorded on the engine stream around the pa_decode call."""
        ids = self._ids_for(seqs)
        n = len(ids)
        q = to_device_rows(q, self.dtype, self.device)
        if out is None:
            out = torch.empty_like(q)
        i = self._stage()
        buf = self._pin_np[i]
        lens, tables = buf[:n], buf[n:n + n * self.max_blocks].reshape(n, self.max_blocks)
        self.bm.block_tables_into(ids, self.max_blocks, tables, lens)
        dev = self._upload(i, n + n * self.max_blocks)
        p = self._decode_params(tables, params)
        if events is not None:
            events[0].record(self._stream())
        pa_decode(q, self.k_cache, self.v_cache, dev[n:n + n * self.max_blocks].view(n, self.max_blocks),
                  dev[:n], scale, out, stream=self._stream(), params=p)
        if events is not None:
            events[1].record(self._stream())
        return out

    def decode_step(self, seqs, k_rows, v_rows, q, scale: float, out=None, params=None, events=None):
        """append + attend: the whole hot path of one step.

        Without ``events`` the whole host side runs in libpa (pa_step_decode: block-manager
        step, tables staged in mapped pinned memory, copies, an append that also carries the
        staged tables to the device, decode).  ``events`` (start, end):
        CUDA events recorded on the engine stream around the pa_decode call (decode kernel +
        merge), for timing; the step then runs through the separate calls.
        Returns (out, number of copy-on-write pairs, context lengths).
        """
        ids = self._ids_for(seqs)
        n = len(ids)
        if events is None:
            if out is None:
                out = torch.empty_like(q)
            ring = self._step_lens[self._k % len(self._step_lens)]
            self._k += 1
            lens = ring[:n] if n <= ring.shape[0] else np.empty(n, np.int32)
            nc = pa_step_decode(self.bm, ids, self.max_blocks, k_rows, v_rows, q, self.k_cache, self.v_cache, scale,
                                out, params=params, auto_share=self.auto_share, stream=self._stream(), lens_out=lens)
            return out, nc, lens
        mb = self.max_blocks
        i = self._stage()
        buf = self._pin_np[i]
        slots, copies = buf[:n], buf[n:3 * n].reshape(n, 2)
        lens = buf[3 * n:4 * n]
        tables = buf[4 * n:4 * n + n * mb].reshape(n, mb)
        nc = self.bm.step_into(ids, slots, copies)
        self.bm.block_tables_into(ids, mb, tables, lens)
        dev = self._upload(i, 4 * n + n * mb)
        st = self._stream()
        if nc:
            pa_copy_blocks(self.k_cache, self.v_cache, dev[n:n + 2 * nc].view(nc, 2), stream=st)
        pa_cache_append(k_rows, v_rows, dev[:n], self.k_cache, self.v_cache, stream=st)
        if out is None:
            out = torch.empty_like(q)
        if events is not None:
            events[0].record(st)
        pa_decode(q, self.k_cache, self.v_cache, dev[4 * n:4 * n + n * mb].view(n, mb), dev[3 * n:4 * n],
                  scale, out, stream=st, params=self._decode_params(tables, params))
        if events is not None:
            events[1].record(st)
        return out, nc, lens


def run_workload_ops(engine: PagedKVEngine, w, attend_params=None):
    """Replay a workload op list through the engine. Returns ({attend / prefill op
    index: out}, trace); token-driven admissions record ``trace["n_cached"][seq]``."""
    outs = {}
    trace = {"n_cached": {}}
    for i, op in enumerate(w.ops):
        kind = op[0]
        if kind == "add":
            k, v = w.rows(i)
            trace[i] = {"slots": engine.add_seq(op[1], k, v).tolist(), "copies": []}
        elif kind == "fork":
            engine.fork(op[1], op[2])
        elif kind == "step":
            k, v = w.rows(i)
            slots, copies = engine.step(op[1], k, v)
            trace[i] = {"slots": slots.tolist(), "copies": [tuple(c) for c in copies.tolist()]}
        elif kind == "free":
            engine.free(op[1])
        elif kind == "extend":
            k, v = w.rows(i)
            slots, copies = engine.extend(op[1], k, v)
            trace[i] = {"slots": slots.tolist(), "copies": [tuple(c) for c in copies.tolist()]}
        elif kind == "prefill":
            outs[i] = engine.prefill(op[1], op[2], w.query(i), w.scale)
        elif kind == "add_tokens":
            n_cached, slots = engine.add_seq_cached(op[1], op[2])
            trace["n_cached"][op[1]] = n_cached
            trace[i] = {"slots": slots.tolist(), "copies": [], "n_cached": n_cached}
            if len(slots):
                k, v = w.token_rows(i)
                engine.write_rows(slots, k[n_cached:], v[n_cached:])
        elif kind in ("extend_tokens", "step_tokens"):
            k, v = w.token_rows(i)
            if kind == "extend_tokens":
                slots, copies = engine.extend_tokens(op[1], op[2], k, v)
            else:
                slots, copies = engine.step_tokens(op[1], op[2], k, v)
            trace[i] = {"slots": slots.tolist(), "copies": [tuple(c) for c in copies.tolist()]}
        elif kind == "prefill_new":
            seqs = list(op[1])
            lens = [engine.bm.seq_info(s)[0] for s in seqs]
            counts = [lens[j] - trace["n_cached"][s] for j, s in enumerate(seqs)]
            qs = w.position_queries(i)
            q = np.concatenate([qs[j][lens[j] - counts[j]:lens[j]] for j in range(len(seqs))])
            outs[i] = engine.prefill(seqs, counts, q, w.scale)
        elif kind == "attend":
            outs[i] = engine.attend(op[1], w.query(i), w.scale, params=attend_params)
        else:
            raise ValueError(op)
    return outs, trace
