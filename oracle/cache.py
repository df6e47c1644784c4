"""Oracle model of the two paged caches.

Layout from "Solving the LLM Memory Wall" ("The Architecture at a Glance" and the
PagedKVCache of "Implementation"): separate K and V tensors, each
[num_blocks, block_size, heads, head_dim].  A token row is written at
[frame, offset] = the flat slot frame*B + offset of the [num_blocks*B, heads,
head_dim] view; copy-on-write copies a whole frame.

Storage is the workload's storage dtype (float32, float16, or bf16 bit patterns in
uint16).  A model may keep only a subset of frames (``keep``): writes and copies
into other frames are dropped, which is exact for every kept frame as long as the
subset is closed under copy sources.
"""

from __future__ import annotations

import numpy as np

_NP = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}


def decode_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage values -> float64 (exact for all three storage types)."""
    if dtype == "bf16":
        wide = a.astype(np.uint32) << np.uint32(16)
        return wide.view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class OracleKVCache:
    def __init__(self, num_blocks, block_size, num_heads, head_dim, dtype, keep=None):
        self.num_blocks, self.block_size = num_blocks, block_size
        self.num_heads, self.head_dim, self.dtype = num_heads, head_dim, dtype
        self.keep = None if keep is None else sorted(set(int(b) for b in keep))
        if self.keep is None:
            shape = (num_blocks, block_size, num_heads, head_dim)
            self.k = np.zeros(shape, _NP[dtype])
            self.v = np.zeros(shape, _NP[dtype])
        else:
            self.k = {b: np.zeros((block_size, num_heads, head_dim), _NP[dtype]) for b in self.keep}
            self.v = {b: np.zeros((block_size, num_heads, head_dim), _NP[dtype]) for b in self.keep}

    def write(self, slots, k_rows, v_rows) -> None:
        """k/v rows [T, H, D] into the given flat slots (negative slot = padding, skipped)."""
        B = self.block_size
        for t, slot in enumerate(slots):
            if slot < 0:
                continue
            frame, offset = divmod(int(slot), B)
            if self.keep is None:
                self.k[frame, offset] = k_rows[t]
                self.v[frame, offset] = v_rows[t]
            elif frame in self.k:
                self.k[frame][offset] = k_rows[t]
                self.v[frame][offset] = v_rows[t]

    def copy_block(self, src: int, dst: int) -> None:
        if self.keep is None:
            self.k[dst] = self.k[src]
            self.v[dst] = self.v[src]
        elif dst in self.k:
            self.k[dst] = self.k[src].copy()
            self.v[dst] = self.v[src].copy()

    def frame(self, which: str, b: int) -> np.ndarray:
        arr = self.k if which == "k" else self.v
        return arr[b]


def split_layout(k: np.ndarray, v: np.ndarray, elem_bytes: int):
    """The kernel-side cache layout of "PagedAttention: Virtual Memory Guide for LLM
    Inference", "3. PagedAttention CUDA Kernel Execution" (the conceptual kernel
    signature): K as [num_blocks, heads, head_dim/x, block_size, x] and V as
    [num_blocks, heads, head_dim, block_size], x = elements per 16 bytes, holding the
    same values as the [num_blocks, block_size, heads, head_dim] caches."""
    nb, B, H, D = k.shape
    x = 16 // elem_bytes
    ks = k.reshape(nb, B, H, D // x, x).transpose(0, 2, 3, 1, 4)
    vs = v.transpose(0, 2, 3, 1)
    return np.ascontiguousarray(ks), np.ascontiguousarray(vs)
