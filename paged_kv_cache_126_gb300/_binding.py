"""Thin ctypes binding of libpa (include/pa.h): argument marshalling only.

Every device operation runs in libpa's CUDA kernels; this module turns torch
tensors into ``pa_tensor`` descriptors and return codes into exceptions.  If
``libpa.so`` is missing the import fails: there is no fallback path.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

PA_F32, PA_F16, PA_BF16, PA_I32 = 0, 1, 2, 3
PA_OK = 0
PA_WARN_DOUBLE_FREE = 1
PA_ERR_INVALID = -1
PA_ERR_OUT_OF_BLOCKS = -6
PA_ERR_UNKNOWN_SEQ = -7
PA_ERR_SEQ_EXISTS = -8
PA_ERR_SCRATCH_LIMIT = -12
PA_ERR_HOST_MEMORY = -13
PA_ERR_UNSUPPORTED = -10
PA_ERR_CAPACITY = -11

PA_DEV_BAD_SLOT = 0x1
PA_DEV_BAD_BLOCK = 0x2
PA_DEV_BAD_LEN = 0x4
PA_DEV_BAD_COPY = 0x8
PA_DEV_TIMEOUT = 0x10

_TORCH_DT = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.int32: PA_I32}


class PaTensor(C.Structure):
    _fields_ = [("data", C.c_void_p), ("dtype", C.c_int32), ("ndim", C.c_int32),
                ("shape", C.c_int64 * 4), ("stride", C.c_int64 * 4)]


class PaDecodeParams(C.Structure):
    _fields_ = [("partition_tokens", C.c_int32), ("heads_per_cta", C.c_int32),
                ("warps_per_head", C.c_int32), ("stages", C.c_int32), ("ctas_per_sm", C.c_int32),
                ("items_per_cta", C.c_int32), ("generic_only", C.c_int32), ("share_prefix", C.c_int32)]


class PaBmUsage(C.Structure):
    _fields_ = [(name, C.c_int64) for name in (
        "num_seqs", "frames_total", "frames_in_use", "frames_cached", "table_entries", "tokens_logical",
        "slots_filled", "max_seq_waste")]


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libpa.so not found at {_LIB_PATH}; build it first "
                          "(python paged_kv_cache_126_gb300/build.py)")
    lib = C.CDLL(_LIB_PATH)
    P = C.POINTER(PaTensor)
    # int32 / int64 array arguments travel as plain addresses (numpy's .ctypes.data): a
    # typed pointer built with .ctypes.data_as costs over a microsecond more per array
    i32p = i64p = C.c_void_p
    vp = C.c_void_p
    sig = {
        "pa_cache_append": ([P, P, P, P, P, vp], C.c_int),
        "pa_copy_blocks": ([P, P, P, vp], C.c_int),
        "pa_decode": ([P, P, P, P, P, C.c_float, P, vp], C.c_int),
        "pa_decode_ex": ([P, P, P, P, P, C.c_float, P, C.POINTER(PaDecodeParams), vp], C.c_int),
        "pa_decode_static": ([P, P, P, P, P, C.c_float, P, vp], C.c_int),
        "pa_prefill": ([P, P, P, P, P, P, C.c_float, P, vp], C.c_int),
        "pa_cache_append_split": ([P, P, P, P, P, vp], C.c_int),
        "pa_decode_split": ([P, P, P, P, P, C.c_float, P, vp], C.c_int),
        "pa_get_device_status": ([vp, i32p], C.c_int),
        "pa_strerror": ([C.c_int], C.c_char_p),
        "pa_launch_count": ([], C.c_int64),
        "pa_shutdown": ([], C.c_int),
        "pa_bm_create": ([C.c_int32, C.c_int32, i32p, C.POINTER(vp)], C.c_int),
        "pa_bm_destroy": ([vp], None),
        "pa_bm_add_seq": ([vp, C.c_int64, C.c_int32, i32p], C.c_int),
        "pa_bm_append": ([vp, C.c_int64, i32p, i32p, i32p], C.c_int),
        "pa_bm_step": ([vp, i64p, C.c_int32, i32p, i32p, i32p], C.c_int),
        "pa_bm_extend": ([vp, C.c_int64, C.c_int32, i32p, i32p, i32p], C.c_int),
        "pa_bm_fork": ([vp, C.c_int64, C.c_int64], C.c_int),
        "pa_step_decode": ([vp, i64p, C.c_int32, C.c_int32, P, P, P, P, P, C.c_float, P,
                            C.POINTER(PaDecodeParams), C.c_int32, vp, i32p, i32p], C.c_int),
        "pa_bm_fork_many": ([vp, i64p, i64p, C.c_int32], C.c_int),
        "pa_bm_free_many": ([vp, i64p, C.c_int32], C.c_int),
        "pa_bm_free": ([vp, C.c_int64], C.c_int),
        "pa_bm_block_tables": ([vp, i64p, C.c_int32, C.c_int32, i32p, i32p], C.c_int),
        "pa_bm_seq_info": ([vp, C.c_int64, i32p, i32p], C.c_int),
        "pa_bm_table": ([vp, C.c_int64, i32p, C.c_int32, i32p], C.c_int),
        "pa_bm_slot": ([vp, C.c_int64, C.c_int32, i32p], C.c_int),
        "pa_bm_num_free": ([vp, i32p], C.c_int),
        "pa_bm_free_list": ([vp, i32p, C.c_int32, i32p], C.c_int),
        "pa_bm_ref_counts": ([vp, i32p, C.c_int32], C.c_int),
        "pa_bm_num_seqs": ([vp, i32p], C.c_int),
        "pa_bm_add_seq_cached": ([vp, C.c_int64, i32p, C.c_int32, i32p, i32p], C.c_int),
        "pa_bm_step_tokens": ([vp, i64p, i32p, C.c_int32, i32p, i32p, i32p], C.c_int),
        "pa_bm_extend_tokens": ([vp, C.c_int64, i32p, C.c_int32, i32p, i32p, i32p], C.c_int),
        "pa_bm_cached_frames": ([vp, i32p, C.c_int32, i32p], C.c_int),
        "pa_bm_usage": ([vp, C.POINTER(PaBmUsage)], C.c_int),
        "pa_bm_export": ([vp, i64p, i32p, i64p, i32p, i32p, i32p, C.c_int32, C.c_int64, i32p, i64p, i32p], C.c_int),
        "pa_selftest_wait_timeout": ([i64p, vp], C.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


LIB = _load()
EXPORTED = (
    "pa_cache_append", "pa_copy_blocks", "pa_decode", "pa_decode_ex", "pa_decode_static", "pa_prefill",
    "pa_cache_append_split", "pa_decode_split",
    "pa_get_device_status",
    "pa_strerror", "pa_launch_count", "pa_shutdown", "pa_bm_create", "pa_bm_destroy", "pa_bm_add_seq",
    "pa_bm_append", "pa_bm_step", "pa_bm_extend", "pa_bm_fork", "pa_bm_free", "pa_bm_block_tables", "pa_bm_seq_info",
    "pa_bm_table", "pa_bm_slot", "pa_bm_num_free", "pa_bm_free_list", "pa_bm_ref_counts",
    "pa_bm_num_seqs", "pa_bm_add_seq_cached", "pa_bm_step_tokens", "pa_bm_extend_tokens", "pa_bm_cached_frames",
    "pa_bm_fork_many", "pa_bm_free_many", "pa_step_decode", "pa_bm_usage", "pa_selftest_wait_timeout",
    "pa_bm_export",
)


def strerror(code: int) -> str:
    """Message of a libpa return code (``pa_strerror``)."""
    return LIB.pa_strerror(int(code)).decode()


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise PAError(rc, where)
    return rc


_DESC_CACHE: dict = {}


def tensor_desc(t: torch.Tensor) -> PaTensor:
    """pa_tensor describing a torch tensor (no copy).

    Descriptors are cached by their whole content (address, dtype, shape, strides): the
    library only reads them, and building one costs several microseconds of Python, a
    visible share of a decode step's host time."""
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _DESC_CACHE.get(key)
    if d is not None:
        return d
    d = _make_desc(t)
    if len(_DESC_CACHE) >= 4096:
        _DESC_CACHE.clear()
    _DESC_CACHE[key] = d
    return d


def _make_desc(t: torch.Tensor) -> PaTensor:
    # every pa_tensor argument is device memory: a host tensor would hand the kernels a
    # host address (checked here, once per distinct tensor: descriptors are cached)
    if not t.is_cuda:
        raise ValueError("device operations take CUDA tensors")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device} but the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype not in _TORCH_DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() < 1 or t.dim() > 4:
        raise ValueError("tensors must have 1..4 dims")
    d = PaTensor()
    d.data = t.data_ptr() or None
    d.dtype = _TORCH_DT[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream_of(t: torch.Tensor, stream):
    if not t.is_cuda:
        raise ValueError("device operations take CUDA tensors")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device} but the current device is cuda:{torch.cuda.current_device()}")
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return C.c_void_p(s.cuda_stream)


def _ref(d: PaTensor):
    return C.byref(d)


def pa_cache_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """``pa_cache_append``: k_new / v_new rows [T, H, D] into the caches at slot_mapping [T] (int32; < 0 skipped)."""
    st = _stream_of(k_cache, stream)
    ds = [tensor_desc(t) for t in (k_new, v_new, slot_mapping, k_cache, v_cache)]
    _check(LIB.pa_cache_append(*map(_ref, ds), st), "pa_cache_append")


def pa_copy_blocks(k_cache, v_cache, pairs, stream=None) -> None:
    """``pa_copy_blocks``: whole-frame copies (src, dst) for copy-on-write, K and V caches."""
    st = _stream_of(k_cache, stream)
    ds = [tensor_desc(t) for t in (k_cache, v_cache, pairs)]
    _check(LIB.pa_copy_blocks(*map(_ref, ds), st), "pa_copy_blocks")


def make_params(params) -> PaDecodeParams | None:
    """A ``pa_decode_params`` from a dict of launch options (unknown keys raise ValueError; 0 = automatic)."""
    if params is None:
        return None
    if isinstance(params, PaDecodeParams):
        return params
    p = PaDecodeParams()
    names = {f[0] for f in PaDecodeParams._fields_}
    for k, v in dict(params).items():
        if k not in names:
            raise ValueError(f"unknown decode option {k!r}")
        setattr(p, k, int(v))
    return p


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None, params=None):
    """``pa_decode`` (or ``pa_decode_ex`` when ``params`` is given): decode attention into ``out`` [S, H, D]."""
    st = _stream_of(q, stream)
    ds = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, context_lens)]
    o = tensor_desc(out)
    p = make_params(params)
    if p is None:
        rc = LIB.pa_decode(*map(_ref, ds), C.c_float(scale), C.byref(o), st)
    else:
        rc = LIB.pa_decode_ex(*map(_ref, ds), C.c_float(scale), C.byref(o), C.byref(p), st)
    _check(rc, "pa_decode")
    return out


def pa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out, params=None, stream=None):
    """``pa_decode_ex``: ``pa_decode`` with explicit launch options (a dict, see ``make_params``)."""
    return pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=stream,
                     params=params or {})


def pa_step_decode(bm, seq_ids, max_blocks, k_new, v_new, q, k_cache, v_cache, scale, out, params=None,
                   auto_share=True, stream=None, lens_out=None) -> int:
    """One decode step with the host side in libpa (see include/pa.h): block-manager step,
    tables, one staged upload, copy-on-write copies, append and decode.  seq_ids: int64
    host array; lens_out: optional int32 host array of len(seq_ids) for the context
    lengths.  Returns the number of copy-on-write frame copies."""
    st = _stream_of(q, stream)
    ids = seq_ids if isinstance(seq_ids, np.ndarray) and seq_ids.dtype == np.int64 else \
        np.ascontiguousarray(seq_ids, dtype=np.int64)
    ds = [tensor_desc(t) for t in (k_new, v_new, q, k_cache, v_cache)]
    o = tensor_desc(out)
    p = make_params(params)
    nc = C.c_int32()
    _check(LIB.pa_step_decode(bm._h, _i64(ids), len(ids), int(max_blocks), *map(_ref, ds), C.c_float(scale),
                              C.byref(o), C.byref(p) if p is not None else None, int(bool(auto_share)), st,
                              C.byref(nc), _i32(lens_out) if lens_out is not None else None), "pa_step_decode")
    return nc.value


def pa_decode_static(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None):
    """pa_decode without any device allocation: scratch comes from a fixed 16 MiB array
    inside libpa (for callers whose device memory belongs to their own allocator).
    Calls must not overlap on the GPU; see include/pa.h."""
    st = _stream_of(q, stream)
    ds = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, context_lens)]
    o = tensor_desc(out)
    _check(LIB.pa_decode_static(*map(_ref, ds), C.c_float(scale), C.byref(o), st), "pa_decode_static")
    return out


def pa_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, out, stream=None):
    """Causal attention for query chunks (see include/pa.h)."""
    st = _stream_of(q, stream)
    ds = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, context_lens, query_start)]
    o = tensor_desc(out)
    _check(LIB.pa_prefill(*map(_ref, ds), C.c_float(scale), C.byref(o), st), "pa_prefill")
    return out


def pa_cache_append_split(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """Cache append into the split layout (see include/pa.h); k_cache is the 4-D view
    [num_blocks, H, D/8, B*8] of [num_blocks, H, D/8, B, 8]."""
    st = _stream_of(k_new, stream)
    ds = [tensor_desc(t) for t in (k_new, v_new, slot_mapping, k_cache, v_cache)]
    _check(LIB.pa_cache_append_split(*map(_ref, ds), st), "pa_cache_append_split")


def pa_decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None):
    """Decode attention over the split layout (see include/pa.h)."""
    st = _stream_of(q, stream)
    ds = [tensor_desc(t) for t in (q, k_cache, v_cache, block_tables, context_lens)]
    o = tensor_desc(out)
    _check(LIB.pa_decode_split(*map(_ref, ds), C.c_float(scale), C.byref(o), st), "pa_decode_split")
    return out


def pa_get_device_status(stream=None) -> int:
    """``pa_get_device_status``: synchronise the stream, return and clear the sticky PA_DEV_* bits."""
    s = stream if stream is not None else torch.cuda.current_stream()
    v = C.c_int32(0)
    _check(LIB.pa_get_device_status(C.c_void_p(s.cuda_stream), C.byref(v)), "pa_get_device_status")
    return v.value


def pa_selftest_wait_timeout(stream=None) -> list:
    """Run the bounded-wait self-test (about 2 s): [first wait ok, second wait ok,
    cycles of the first, cycles of the second]."""
    s = stream if stream is not None else torch.cuda.current_stream()
    res = np.zeros(4, np.int64)
    _check(LIB.pa_selftest_wait_timeout(res.ctypes.data_as(C.POINTER(C.c_int64)), C.c_void_p(s.cuda_stream)),
           "pa_selftest_wait_timeout")
    return res.tolist()


def pa_launch_count() -> int:
    """Kernels libpa has launched in this process (``pa_launch_count``)."""
    return int(LIB.pa_launch_count())


def pa_shutdown() -> None:
    """``pa_shutdown``: free the library-owned workspaces and staging rings."""
    _check(LIB.pa_shutdown(), "pa_shutdown")


def _i32(a: np.ndarray):
    """Address of an int32 array's data (the callee's int32_t* argument)."""
    if a.dtype != np.int32:
        raise TypeError(f"expected an int32 array, got {a.dtype}")
    return a.ctypes.data


def _i64(a: np.ndarray):
    """Address of an int64 array's data (the callee's int64_t* argument)."""
    if a.dtype != np.int64:
        raise TypeError(f"expected an int64 array, got {a.dtype}")
    return a.ctypes.data


class BlockManager:
    """Host block manager of libpa (free list, refcounts, fork, copy-on-write, prefix cache)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        h = C.c_void_p()
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            if self._order.shape != (self.num_blocks,):
                raise ValueError("free_order must list every block id once")
            order = _i32(self._order)
        _check(LIB.pa_bm_create(self.num_blocks, self.block_size, order, C.byref(h)), "pa_bm_create")
        self._h = h

    def close(self) -> None:
        """Destroy the native manager (``pa_bm_destroy``); later calls are invalid."""
        if self._h:
            LIB.pa_bm_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        """The opaque ``pa_bm*`` for direct C calls."""
        return self._h

    def add_seq(self, seq: int, num_tokens: int) -> np.ndarray:
        """``pa_bm_add_seq``: frames for a prompt of num_tokens (all-or-nothing); returns its slots."""
        slots = np.empty(max(int(num_tokens), 1), np.int32)
        _check(LIB.pa_bm_add_seq(self._h, int(seq), int(num_tokens), _i32(slots)), "pa_bm_add_seq")
        return slots[: int(num_tokens)]

    def append(self, seq: int):
        """``pa_bm_append``: one token; returns (slot, (src, dst) copy or None)."""
        slot, src, dst = C.c_int32(), C.c_int32(), C.c_int32()
        _check(LIB.pa_bm_append(self._h, int(seq), C.byref(slot), C.byref(src), C.byref(dst)), "pa_bm_append")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def step_into(self, ids: np.ndarray, slots_out: np.ndarray, copies_out: np.ndarray) -> int:
        """One decode step; fills caller arrays, returns the number of copy pairs."""
        nc = C.c_int32(0)
        _check(LIB.pa_bm_step(self._h, _i64(ids), len(ids), _i32(slots_out), _i32(copies_out), C.byref(nc)),
               "pa_bm_step")
        return nc.value

    def step(self, seqs):
        """``pa_bm_step``: one token for each listed sequence in order (all-or-nothing); returns (slots, copies [k, 2])."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        slots = np.empty(max(len(ids), 1), np.int32)
        copies = np.empty((max(len(ids), 1), 2), np.int32)
        n = self.step_into(ids, slots, copies)
        return slots[: len(ids)], copies[:n]

    def extend(self, seq: int, n: int):
        """n new tokens for one sequence (a prompt chunk). Returns (slots, copies)."""
        n = int(n)
        slots = np.empty(max(n, 1), np.int32)
        copies = np.empty((max(n, 1), 2), np.int32)
        nc = C.c_int32(0)
        _check(LIB.pa_bm_extend(self._h, int(seq), n, _i32(slots), _i32(copies), C.byref(nc)), "pa_bm_extend")
        return slots[:n], copies[: nc.value]

    # -- prefix caching -------------------------------------------------------------
    def add_seq_cached(self, seq: int, tokens):
        """Admit a prompt by its token ids; returns (n_cached, slots of the uncached tokens)."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        L = len(toks)
        slots = np.empty(max(L, 1), np.int32)
        nc = C.c_int32(0)
        _check(LIB.pa_bm_add_seq_cached(self._h, int(seq), _i32(toks) if L else None, L, _i32(slots),
                                        C.byref(nc)), "pa_bm_add_seq_cached")
        return nc.value, slots[: L - nc.value]

    def step_tokens(self, seqs, tokens):
        """``pa_bm_step_tokens``: ``step`` with the new tokens' ids (prefix-cache registration)."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        n = len(ids)
        if len(toks) != n:
            raise ValueError("one token id per appended sequence")
        slots = np.empty(max(n, 1), np.int32)
        copies = np.empty((max(n, 1), 2), np.int32)
        nc = C.c_int32(0)
        _check(LIB.pa_bm_step_tokens(self._h, _i64(ids), _i32(toks), n, _i32(slots), _i32(copies), C.byref(nc)),
               "pa_bm_step_tokens")
        return slots[:n], copies[: nc.value]

    def extend_tokens(self, seq: int, tokens):
        """``pa_bm_extend_tokens``: a chunk of tokens with their ids; returns (slots, copies)."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        n = len(toks)
        slots = np.empty(max(n, 1), np.int32)
        copies = np.empty((max(n, 1), 2), np.int32)
        nc = C.c_int32(0)
        _check(LIB.pa_bm_extend_tokens(self._h, int(seq), _i32(toks) if n else None, n, _i32(slots), _i32(copies),
                                       C.byref(nc)), "pa_bm_extend_tokens")
        return slots[:n], copies[: nc.value]

    def cached_frames(self) -> list:
        """``pa_bm_cached_frames``: 1 for each frame holding a registered block, else 0."""
        out = np.empty(self.num_blocks, np.int32)
        n = C.c_int32()
        _check(LIB.pa_bm_cached_frames(self._h, _i32(out), self.num_blocks, C.byref(n)), "pa_bm_cached_frames")
        return out.tolist()

    def fork(self, parent: int, child: int) -> None:
        """``pa_bm_fork``: child shares every frame of parent (zero-copy)."""
        _check(LIB.pa_bm_fork(self._h, int(parent), int(child)), "pa_bm_fork")

    def free(self, seq: int) -> int:
        """``pa_bm_free``: release a sequence; returns PA_WARN_DOUBLE_FREE if it was not live."""
        return _check(LIB.pa_bm_free(self._h, int(seq)), "pa_bm_free")

    def fork_many(self, parents, children) -> None:
        """``pa_bm_fork_many``: forks in order, all-or-nothing (a child may be a later parent)."""
        p = np.ascontiguousarray(parents, dtype=np.int64)
        c = np.ascontiguousarray(children, dtype=np.int64)
        if p.shape != c.shape or p.ndim != 1:
            raise ValueError("parents and children must be 1-D and of equal length")
        _check(LIB.pa_bm_fork_many(self._h, _i64(p), _i64(c), len(p)), "pa_bm_fork_many")

    def free_many(self, seqs) -> int:
        """``pa_bm_free_many``: frees in order; PA_WARN_DOUBLE_FREE if any id was not live."""
        s = np.ascontiguousarray(seqs, dtype=np.int64)
        return _check(LIB.pa_bm_free_many(self._h, _i64(s), len(s)), "pa_bm_free_many")

    def block_tables_into(self, ids: np.ndarray, max_blocks: int, tables_out: np.ndarray, lens_out: np.ndarray):
        """``pa_bm_block_tables`` into caller arrays: tables [n, max_blocks] (-1 padded), lens [n]."""
        _check(LIB.pa_bm_block_tables(self._h, _i64(ids), len(ids), int(max_blocks), _i32(tables_out),
                                      _i32(lens_out)), "pa_bm_block_tables")

    def block_tables(self, seqs, max_blocks: int):
        """``pa_bm_block_tables``: (tables [n, max_blocks] int32, lens [n] int32) for the listed sequences."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        tables = np.empty((max(len(ids), 1), max(int(max_blocks), 1)), np.int32)
        lens = np.empty(max(len(ids), 1), np.int32)
        self.block_tables_into(ids, max_blocks, tables, lens)
        return tables[: len(ids), : int(max_blocks)], lens[: len(ids)]

    def seq_info(self, seq: int):
        """``pa_bm_seq_info``: (length, number of frames) of a live sequence."""
        L, nb = C.c_int32(), C.c_int32()
        _check(LIB.pa_bm_seq_info(self._h, int(seq), C.byref(L), C.byref(nb)), "pa_bm_seq_info")
        return L.value, nb.value

    def table(self, seq: int) -> list:
        """``pa_bm_table``: the frame ids of a live sequence, in order."""
        _, nb = self.seq_info(seq)
        out = np.empty(max(nb, 1), np.int32)
        n = C.c_int32()
        _check(LIB.pa_bm_table(self._h, int(seq), _i32(out), nb, C.byref(n)), "pa_bm_table")
        return out[: n.value].tolist()

    def slot(self, seq: int, pos: int) -> int:
        """``pa_bm_slot``: flat slot (frame * B + offset) of token ``pos`` of a live sequence."""
        s = C.c_int32()
        _check(LIB.pa_bm_slot(self._h, int(seq), int(pos), C.byref(s)), "pa_bm_slot")
        return s.value

    @property
    def num_free(self) -> int:
        """``pa_bm_num_free``: frames on the free list."""
        n = C.c_int32()
        _check(LIB.pa_bm_num_free(self._h, C.byref(n)), "pa_bm_num_free")
        return n.value

    def free_list(self) -> list:
        """``pa_bm_free_list``: the free list, front (next to be handed out) first."""
        out = np.empty(self.num_blocks, np.int32)
        n = C.c_int32()
        _check(LIB.pa_bm_free_list(self._h, _i32(out), self.num_blocks, C.byref(n)), "pa_bm_free_list")
        return out[: n.value].tolist()

    def ref_counts(self) -> list:
        """``pa_bm_ref_counts``: reference count of every frame."""
        out = np.empty(self.num_blocks, np.int32)
        _check(LIB.pa_bm_ref_counts(self._h, _i32(out), self.num_blocks), "pa_bm_ref_counts")
        return out.tolist()

    @property
    def num_seqs(self) -> int:
        """``pa_bm_num_seqs``: live sequences."""
        n = C.c_int32()
        _check(LIB.pa_bm_num_seqs(self._h, C.byref(n)), "pa_bm_num_seqs")
        return n.value

    def export(self) -> dict:
        """Whole state (``pa_bm_export``): {"tables": {seq: [frames]}, "lens": {seq: len},
        "free": [front first], "refs": [per frame]}."""
        ns, ne, nf = C.c_int32(), C.c_int64(), C.c_int32()
        dummy64, dummy32 = np.zeros(1, np.int64), np.zeros(1, np.int32)
        free = np.empty(self.num_blocks, np.int32)
        refs = np.empty(self.num_blocks, np.int32)
        rc = LIB.pa_bm_export(self._h, _i64(dummy64), _i32(dummy32),
                              _i64(dummy64), None, _i32(free), _i32(refs), 0, 0,
                              C.byref(ns), C.byref(ne), C.byref(nf))
        if rc not in (PA_OK, PA_ERR_CAPACITY):
            _check(rc, "pa_bm_export")
        n, e = ns.value, ne.value
        ids, lens = np.empty(max(n, 1), np.int64), np.empty(max(n, 1), np.int32)
        offs, tabs = np.empty(n + 1, np.int64), np.empty(max(e, 1), np.int32)
        _check(LIB.pa_bm_export(self._h, _i64(ids), _i32(lens), _i64(offs),
                                _i32(tabs), _i32(free), _i32(refs), n, e, C.byref(ns), C.byref(ne), C.byref(nf)),
               "pa_bm_export")
        return {"tables": {int(ids[i]): tabs[offs[i]:offs[i + 1]].tolist() for i in range(n)},
                "lens": {int(ids[i]): int(lens[i]) for i in range(n)},
                "free": free[: nf.value].tolist(), "refs": refs.tolist()}

    def usage(self) -> dict:
        """Memory accounting of the pool (``pa_bm_usage``): field name -> count."""
        u = PaBmUsage()
        _check(LIB.pa_bm_usage(self._h, C.byref(u)), "pa_bm_usage")
        return {name: int(getattr(u, name)) for name, _ in PaBmUsage._fields_}
