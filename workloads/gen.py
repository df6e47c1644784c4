"""Workload definitions and seeded draws.

A workload is a list of operations on a paged KV cache plus the random payload
each operation carries:

* ``("add", seq, n)``     -- a new sequence with an ``n``-token prompt; the op's
                             payload is ``n`` K rows and ``n`` V rows.
* ``("fork", parent, child)`` -- the child shares the parent's blocks.
* ``("step", seqs)``      -- one decode step: one new token for each listed
                             sequence, in list order; payload: ``len(seqs)`` rows.
* ``("attend", seqs)``    -- single-query decode attention for each listed
                             sequence; payload: one query per sequence.
* ``("free", seq)``       -- the sequence finishes.
* ``("extend", seq, n)``  -- a prompt chunk: n new tokens for one sequence; payload:
                             n K rows and n V rows.
* ``("prefill", seqs, counts)`` -- causal attention for the last counts[i] positions
                             of seqs[i]; payload: sum(counts) queries, grouped by
                             sequence in list order.

Token-driven ops (prefix caching).  Their K/V rows are a function of the token
prefix, as a model's would be: the row of position j is drawn from a stream keyed
by a 64-bit identity of tokens 0..j, so two requests with the same prefix carry
identical rows for it.

* ``("add_tokens", seq, tokens)``    -- a new sequence given by its token ids.
* ``("extend_tokens", seq, tokens)`` -- tokens appended to one sequence.
* ``("step_tokens", seqs, tokens)``  -- one decode step, tokens[i] for seqs[i].
* ``("prefill_new", seqs)``          -- causal attention for the positions of each
                             sequence that its admission did not find in the cache;
                             payload: queries for every position of each sequence
                             (the consumer takes the ones it needs).

Payloads are drawn from a PCG64 stream keyed by ``(seed, op_index, kind)`` so any
op's rows can be regenerated alone.  Values are drawn as float32 N(0, sigma^2)
and rounded to nearest-even into the storage type; bf16 is carried as uint16 bit
patterns because NumPy has no bf16 type.

Shapes follow the five workloads of the paged-decode study (a 100-block toy
trace, a 64-sequence decode batch, a 4x16k long-context batch, a 16-prompt
parallel-sampling batch with copy-on-write, a 256-sequence serving mix), each with
a scaled-down variant whose oracle finishes in seconds.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "f16", "bf16")
CONFIG_IDS = (0, 1, "1x", 2, 3, 4)

_KIND = {"k": 1, "v": 2, "q": 3}


def storage_numpy_dtype(dtype: str):
    """NumPy type that holds one element of the storage dtype."""
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32, copy=False)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return _bf16_bits(x)
    raise ValueError(dtype)


def random_storage(seed: int, shape, dtype: str, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma) values of the given shape, rounded to the storage dtype (bf16 as
    uint16 bit patterns)."""
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(sigma)
    return _to_storage(x, dtype)


_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on uint64 arrays (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = z + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def prefix_ids(seed: int, tokens) -> np.ndarray:
    """uint64 identity of every token prefix: ids[j] depends on tokens[0..j] only."""
    out = np.empty(len(tokens), np.uint64)
    h = _mix64(np.array([seed], np.uint64))[0]
    with np.errstate(over="ignore"):
        for j, t in enumerate(tokens):
            h = _mix64(np.array([h ^ (np.uint64(int(t) & 0xFFFFFFFF) * np.uint64(0x100000001B3))], np.uint64))[0]
            out[j] = h
    return out


def _keyed_normals(keys: np.ndarray, count: int) -> np.ndarray:
    """float32 [len(keys), count] standard normals, one counter-based stream per key
    (splitmix64 of key and index, Box-Muller on pairs)."""
    keys = np.asarray(keys, np.uint64)
    half = (count + 1) // 2
    idx = np.arange(2 * half, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64(keys[:, None] * np.uint64(0xD1B54A32D192ED03) + idx[None, :])
    u = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    u1, u2 = u[:, 0::2], u[:, 1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    x = np.concatenate([r * np.cos(2 * np.pi * u2), r * np.sin(2 * np.pi * u2)], axis=1)
    return x[:, :count].astype(np.float32)


@dataclass
class Workload:
    name: str
    num_heads: int
    head_dim: int
    block_size: int
    dtype: str
    sigma: float
    num_blocks: int
    free_order: np.ndarray
    ops: list
    seed: int
    # float32 softmax scale handed to the decode call (1/sqrt(head_dim))
    scale: float = field(default=0.0)
    # context length each sequence ends with (for sizing and reporting only)
    final_lens: dict = field(default_factory=dict)

    def __post_init__(self):
        if not self.scale:
            self.scale = float(np.float32(1.0) / np.sqrt(np.float32(self.head_dim)))
        self.free_order = np.asarray(self.free_order, dtype=np.int32)

    # -- payloads ---------------------------------------------------------------
    def _draw(self, op_index: int, kind: str, n: int) -> np.ndarray:
        ss = np.random.SeedSequence([self.seed, op_index, _KIND[kind]])
        g = np.random.Generator(np.random.PCG64(ss))
        x = g.standard_normal(n * self.num_heads * self.head_dim, dtype=np.float32)
        if self.sigma != 1.0:
            x *= np.float32(self.sigma)
        return _to_storage(x, self.dtype).reshape(n, self.num_heads, self.head_dim)

    def rows(self, op_index: int):
        """(k, v) rows carried by an ``add``, ``extend`` or ``step`` op, storage dtype."""
        op = self.ops[op_index]
        n = op[2] if op[0] in ("add", "extend") else len(op[1])
        return self._draw(op_index, "k", n), self._draw(op_index, "v", n)

    def query(self, op_index: int) -> np.ndarray:
        """Queries carried by an ``attend`` op ``[len(seqs), H, D]`` or a ``prefill`` op
        ``[sum(counts), H, D]``, storage dtype."""
        op = self.ops[op_index]
        if op[0] == "attend":
            return self._draw(op_index, "q", len(op[1]))
        assert op[0] == "prefill"
        return self._draw(op_index, "q", int(sum(op[2])))

    # -- token-driven payloads ------------------------------------------------------
    def token_history(self, op_index: int) -> dict:
        """Token ids of every live token-driven sequence just before op ``op_index``."""
        hist = {}
        for op in self.ops[:op_index]:
            kind = op[0]
            if kind == "add_tokens":
                hist[op[1]] = list(op[2])
            elif kind == "extend_tokens":
                hist[op[1]] = hist[op[1]] + list(op[2])
            elif kind == "step_tokens":
                for s, t in zip(op[1], op[2]):
                    hist[s] = hist[s] + [t]
            elif kind == "fork" and op[1] in hist:
                hist[op[2]] = list(hist[op[1]])
            elif kind == "free":
                hist.pop(op[1], None)
        return hist

    def prefix_rows(self, tokens, start: int = 0, stop=None):
        """(k, v) rows [stop-start, H, D] of positions start..stop-1 of a sequence with
        these token ids, storage dtype; each row depends on its token prefix only."""
        stop = len(tokens) if stop is None else stop
        ids = prefix_ids(self.seed, tokens[:stop])[start:stop]
        n, HD = len(ids), self.num_heads * self.head_dim
        x = _keyed_normals(ids, 2 * HD)
        if self.sigma != 1.0:
            x *= np.float32(self.sigma)
        k = _to_storage(x[:, :HD], self.dtype).reshape(n, self.num_heads, self.head_dim)
        v = _to_storage(x[:, HD:], self.dtype).reshape(n, self.num_heads, self.head_dim)
        return k, v

    def token_rows(self, op_index: int):
        """(k, v) rows carried by a token-driven op: every position of an
        ``add_tokens`` prompt, the new positions of ``extend_tokens``, one row per
        sequence of ``step_tokens`` (in op order)."""
        op = self.ops[op_index]
        hist = self.token_history(op_index)
        if op[0] == "add_tokens":
            return self.prefix_rows(list(op[2]))
        if op[0] == "extend_tokens":
            toks = hist[op[1]] + list(op[2])
            return self.prefix_rows(toks, len(hist[op[1]]))
        assert op[0] == "step_tokens"
        ks, vs = [], []
        for s, t in zip(op[1], op[2]):
            toks = hist[s] + [t]
            hist[s] = toks
            k, v = self.prefix_rows(toks, len(toks) - 1)
            ks.append(k)
            vs.append(v)
        return np.concatenate(ks), np.concatenate(vs)

    def position_queries(self, op_index: int):
        """Queries of a ``prefill_new`` op: one array [L_i, H, D] per listed sequence
        (every position of its current length), storage dtype."""
        op = self.ops[op_index]
        hist = self.token_history(op_index)
        out = []
        for i, s in enumerate(op[1]):
            L = len(hist[s])
            ss = np.random.SeedSequence([self.seed, op_index, _KIND["q"], i])
            g = np.random.Generator(np.random.PCG64(ss))
            x = g.standard_normal(L * self.num_heads * self.head_dim, dtype=np.float32)
            if self.sigma != 1.0:
                x *= np.float32(self.sigma)
            out.append(_to_storage(x, self.dtype).reshape(L, self.num_heads, self.head_dim))
        return out

    @property
    def attend_ops(self):
        return [i for i, op in enumerate(self.ops) if op[0] == "attend"]

    @property
    def prefill_ops(self):
        return [i for i, op in enumerate(self.ops) if op[0] == "prefill"]

    @property
    def elem_bytes(self) -> int:
        return {"f32": 4, "f16": 2, "bf16": 2}[self.dtype]


def _pool_size(final_lens, block_size: int, factor: float = 1.2) -> int:
    # Pool sized with headroom over one private block list per sequence.
    need = sum(-(-L // block_size) for L in final_lens)
    return max(1, int(math.ceil(factor * need)))


def _decode_batch(name, lengths, H, D, B, dtype, sigma, seed, *, shuffle=True,
                  pool=None, free_order=None):
    """Prefill ``L-1`` tokens per sequence, one decode step, one attention."""
    lengths = [int(x) for x in lengths]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    nb = pool if pool is not None else _pool_size(lengths, B)
    if free_order is None:
        free_order = rng.permutation(nb).astype(np.int32) if shuffle else np.arange(nb, dtype=np.int32)
    ops = []
    for s, L in enumerate(lengths):
        ops.append(("add", s, max(L - 1, 0)))
    step = tuple(s for s, L in enumerate(lengths) if L >= 1)
    if step:
        ops.append(("step", step))
    ops.append(("attend", tuple(range(len(lengths)))))
    return Workload(name=name, num_heads=H, head_dim=D, block_size=B, dtype=dtype,
                    sigma=sigma, num_blocks=nb, free_order=free_order, ops=ops, seed=seed,
                    final_lens={s: L for s, L in enumerate(lengths)})


def _toy(seed=1000):
    # 100 blocks of 10 token slots, free list 0..99, prompts A:8 B:5 C:12 D:9,
    # then three decode steps, each followed by attention over all four.
    ops = [("add", 0, 8), ("add", 1, 5), ("add", 2, 12), ("add", 3, 9)]
    for _ in range(3):
        ops.append(("step", (0, 1, 2, 3)))
        ops.append(("attend", (0, 1, 2, 3)))
    return Workload(name="toy: 100 blocks x 10 slots, prompts 8/5/12/9 + 3 decode steps",
                    num_heads=2, head_dim=64, block_size=10, dtype="f32", sigma=1.0,
                    num_blocks=100, free_order=np.arange(100, dtype=np.int32), ops=ops,
                    seed=seed, final_lens={0: 11, 1: 8, 2: 15, 3: 12})


def _parallel_sampling(n_prompts, prompt_len, n_branch, r_max, H, D, B, dtype, seed, name):
    """Prompts forked into branches that decode private tokens with copy-on-write.

    Branch 0 of each prompt is the prompt sequence itself; branches 1.. are forks
    taken right after the prompt is added.  Each branch draws r ~ U{0..r_max}
    private tokens; decoding is step-major (prompts in order, branches in order),
    then one attention over every branch.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    r = rng.integers(0, r_max + 1, size=n_prompts * n_branch)
    ops = []
    for p in range(n_prompts):
        base = p * n_branch
        ops.append(("add", base, prompt_len))
        for b in range(1, n_branch):
            ops.append(("fork", base, base + b))
    for k in range(int(r.max()) if len(r) else 0):
        seqs = tuple(s for s in range(n_prompts * n_branch) if r[s] > k)
        ops.append(("step", seqs))
    ops.append(("attend", tuple(range(n_prompts * n_branch))))
    final = {s: prompt_len + int(r[s]) for s in range(n_prompts * n_branch)}
    nb = _pool_size(final.values(), B)
    free_order = rng.permutation(nb).astype(np.int32)
    return Workload(name=name, num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=1.0,
                    num_blocks=nb, free_order=free_order, ops=ops, seed=seed, final_lens=final)


def _log_uniform(rng, n, lo, hi):
    x = np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))).astype(np.int64)
    return np.clip(x, lo, hi)


def build(cfg, small: bool = False) -> Workload:
    """The five workloads (plus the fixed 64x2048 decode batch ``"1x"``).

    ``small=True`` gives a scaled-down variant of the same structure whose oracle
    runs in seconds: several thread-block tiles and a ragged last block remain.
    """
    seed = 1000 + (1 if cfg == "1x" else int(cfg)) + (500 if small else 0)
    if cfg == 0:
        return _toy(seed)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    if cfg == 1:
        if small:
            L = rng.integers(40, 301, size=6)
            return _decode_batch("decode batch (small): 6 seqs, L~U[40,300], H=4, D=128, B=16, f16",
                                 L, 4, 128, 16, "f16", 1.0, seed)
        L = rng.integers(512, 2049, size=64)
        return _decode_batch("decode batch: 64 seqs, L~U[512,2048], H=32, D=128, B=16, f16",
                             L, 32, 128, 16, "f16", 1.0, seed)
    if cfg == "1x":
        S, L = (4, 300) if small else (64, 2048)
        return _decode_batch(f"decode batch: {S} seqs x {L} tokens, H=32, D=128, B=16, f16",
                             [L] * S, 32 if not small else 4, 128, 16, "f16", 1.0, seed)
    if cfg == 2:
        if small:
            return _decode_batch("long context (small): 2 seqs x 2500, H=2, D=128, B=32, bf16",
                                 [2500, 2500], 2, 128, 32, "bf16", 1.0, seed)
        return _decode_batch("long context: 4 seqs x 16384, H=32, D=128, B=32, bf16",
                             [16384] * 4, 32, 128, 32, "bf16", 1.0, seed)
    if cfg == 3:
        if small:
            return _parallel_sampling(3, 100, 4, 40, 2, 128, 16, "f16", seed,
                                      "parallel sampling (small): 3 prompts x 100, 4 branches, r~U{0..40}")
        return _parallel_sampling(16, 1000, 4, 256, 32, 128, 16, "f16", seed,
                                  "parallel sampling: 16 prompts x 1000, 4 branches, r~U{0..256}, H=32, D=128, B=16, f16")
    if cfg == 4:
        if small:
            L = _log_uniform(rng, 24, 16, 800)
            return _decode_batch("serving mix (small): 24 seqs, L~logU[16,800], H=40, D=128, B=16, bf16",
                                 L, 40, 128, 16, "bf16", 0.5, seed)
        L = _log_uniform(rng, 256, 16, 8192)
        return _decode_batch("serving mix: 256 seqs, L~logU[16,8192], H=40, D=128, B=16, bf16",
                             L, 40, 128, 16, "bf16", 0.5, seed)
    raise ValueError(f"unknown workload {cfg!r}")


def chunked_prefill(prefix_lens, chunk_lens, *, H=2, D=128, B=16, dtype="f16", sigma=1.0, seed=11,
                    shuffle=True, name=None) -> Workload:
    """Each sequence has a cached prefix, then one prompt chunk is appended and its
    queries attend causally (a prefill when the prefix is empty)."""
    prefix_lens = [int(x) for x in prefix_lens]
    chunk_lens = [int(x) for x in chunk_lens]
    final = [a + b for a, b in zip(prefix_lens, chunk_lens)]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    nb = _pool_size(final, B)
    free_order = rng.permutation(nb).astype(np.int32) if shuffle else np.arange(nb, dtype=np.int32)
    ops = [("add", s, L) for s, L in enumerate(prefix_lens)]
    ops += [("extend", s, n) for s, n in enumerate(chunk_lens) if n > 0]
    seqs = tuple(range(len(final)))
    ops.append(("prefill", seqs, tuple(chunk_lens)))
    return Workload(name=name or f"chunked prefill: {len(final)} seqs, chunks {chunk_lens[:4]}..., H={H}, D={D}, "
                                 f"B={B}, {dtype}",
                    num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=sigma, num_blocks=nb,
                    free_order=free_order, ops=ops, seed=seed, final_lens={s: L for s, L in enumerate(final)})


def prefill_batch(small: bool = False, dtype: str = "f16") -> Workload:
    """Chunked-prefill batch: 16 sequences, cached prefix ~U{0..3072}, a 512-token
    chunk each (4 sequences, prefix ~U{0..400}, chunks ~U{1..300} when small); fp16
    unless another 16-bit dtype is asked for (same lengths and seeds)."""
    seed = 1010 + (500 if small else 0)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    if small:
        pre = rng.integers(0, 401, size=4)
        ch = rng.integers(1, 301, size=4)
        return chunked_prefill(pre, ch, H=2, D=128, B=16, dtype=dtype, seed=seed,
                               name=f"chunked prefill (small): 4 seqs, prefix~U[0,400], chunk~U[1,300], H=2, "
                                    f"{dtype}")
    pre = rng.integers(0, 3073, size=16)
    return chunked_prefill(pre, [512] * 16, H=32, D=128, B=16, dtype=dtype, seed=seed,
                           name=f"chunked prefill: 16 seqs, prefix~U[0,3072], chunk 512, H=32, D=128, B=16, "
                                f"{dtype}")


def beam_search(n_prompts: int, prompt_len: int, width: int, steps: int, *, H=2, D=128, B=16, dtype="f16",
                sigma=1.0, seed=31, attend_every: int = 1, name=None) -> Workload:
    """Beam search over forked sequences.

    Each prompt is admitted, then forked into ``width`` beams.  Every step appends
    one token to every live beam (prompts in order, beams in order) and, every
    ``attend_every`` steps, attends all of them; then each prompt keeps ``width``
    survivors drawn uniformly with replacement from its beams: a beam drawn c times
    continues and forks c-1 children, a beam never drawn is freed.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    ops, beams, final = [], [], {}
    nid = 0
    for p in range(n_prompts):
        root = nid
        nid += 1
        ops.append(("add", root, prompt_len))
        final[root] = prompt_len
        group = [root]
        for _ in range(width - 1):
            ops.append(("fork", root, nid))
            final[nid] = prompt_len
            group.append(nid)
            nid += 1
        beams.append(group)
    for t in range(steps):
        live = tuple(s for g in beams for s in g)
        ops.append(("step", live))
        for s in live:
            final[s] += 1
        if (t + 1) % attend_every == 0 or t + 1 == steps:
            ops.append(("attend", live))
        if t + 1 == steps:
            break
        for p in range(n_prompts):
            counts = rng.multinomial(width, np.full(width, 1.0 / width))
            new = []
            for beam, c in zip(beams[p], counts):
                if c == 0:
                    ops.append(("free", beam))
                    continue
                new.append(beam)
                for _ in range(int(c) - 1):
                    ops.append(("fork", beam, nid))
                    final[nid] = final[beam]
                    new.append(nid)
                    nid += 1
            beams[p] = new
    per_beam = -(-(steps + B) // B) + 1
    nb = int(math.ceil(1.2 * n_prompts * (-(-prompt_len // B) + 2 * width * per_beam)))
    free_order = rng.permutation(nb).astype(np.int32)
    return Workload(name=name or f"beam search: {n_prompts} prompts x {prompt_len}, width {width}, {steps} steps, "
                                 f"H={H}, D={D}, B={B}, {dtype}",
                    num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=sigma, num_blocks=nb,
                    free_order=free_order, ops=ops, seed=seed, final_lens=final)


def mcts_tree(n_roots: int, prompt_len: int, iterations: int, *, batch: int = 4, rollout_max: int = 24,
              max_nodes: int = 48, H=2, D=128, B=16, dtype="f16", sigma=1.0, seed=41, name=None) -> Workload:
    """Monte Carlo tree search over forked sequences.

    Every iteration picks ``batch`` live nodes at random (with replacement), forks
    each into a new child, extends the child by r ~ U{1..rollout_max} tokens (a
    chunk: copy-on-write of a shared tail, then new frames), and attends all new
    children; while more than ``max_nodes`` nodes live, random non-root nodes are
    freed (their children keep the frames they share).
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    ops, final, live, roots = [], {}, [], set()
    nid = 0
    for _ in range(n_roots):
        ops.append(("add", nid, prompt_len))
        final[nid] = prompt_len
        live.append(nid)
        roots.add(nid)
        nid += 1
    for _ in range(iterations):
        kids = []
        for parent in rng.choice(live, size=batch):
            parent = int(parent)
            ops.append(("fork", parent, nid))
            r = int(rng.integers(1, rollout_max + 1))
            ops.append(("extend", nid, r))
            final[nid] = final[parent] + r
            kids.append(nid)
            nid += 1
        live += kids
        ops.append(("attend", tuple(kids)))
        while len(live) > max_nodes:
            cand = [s for s in live if s not in roots]
            victim = int(rng.choice(cand))
            ops.append(("free", victim))
            live.remove(victim)
    longest = max(final.values())
    nb = int(math.ceil(1.2 * (n_roots * -(-prompt_len // B) + (max_nodes + batch) * (-(-longest // B) - 
                                                                                    prompt_len // B + 2))))
    free_order = rng.permutation(nb).astype(np.int32)
    return Workload(name=name or f"MCTS: {n_roots} roots x {prompt_len}, {iterations} iterations x {batch} "
                                 f"rollouts <= {rollout_max}, <= {max_nodes} nodes, H={H}, D={D}, B={B}, {dtype}",
                    num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=sigma, num_blocks=nb,
                    free_order=free_order, ops=ops, seed=seed, final_lens=final)


def shared_prefix(n_requests: int, system_len: int, user_lens, *, H=2, D=128, B=16, dtype="f16", sigma=1.0,
                  seed=21, turns: int = 1, reply_len: int = 0, free_between: bool = False, pool=None,
                  name=None) -> Workload:
    """Requests that share a system prompt, each followed by a causal prefill of the
    tokens its admission did not find in the cache.

    Request i's prompt is the shared ``system_len`` tokens plus ``user_lens[i]``
    tokens of its own.  With ``turns > 1`` each request then appends a reply of
    ``reply_len`` tokens and returns for another turn as a new sequence whose prompt
    is its whole conversation plus a fresh user message (multi-turn reuse).  With
    ``free_between`` every request of a turn is freed before the next turn is
    admitted (cached frames then come back from the free list).
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    vocab = 1 << 20
    system = rng.integers(0, vocab, size=system_len).tolist()
    user_lens = [int(u) for u in user_lens]
    conv = [system + rng.integers(0, vocab, size=u).tolist() for u in user_lens]
    ops = []
    seq = 0
    final = {}
    live = []
    for t in range(turns):
        ids = []
        for i in range(n_requests):
            ops.append(("add_tokens", seq, tuple(conv[i])))
            ids.append(seq)
            seq += 1
        ops.append(("prefill_new", tuple(ids)))
        for i, s in enumerate(ids):
            final[s] = len(conv[i])
        if t + 1 < turns:
            for i, s in enumerate(ids):
                reply = rng.integers(0, vocab, size=reply_len).tolist()
                if reply:
                    ops.append(("extend_tokens", s, tuple(reply)))
                conv[i] = conv[i] + reply + rng.integers(0, vocab, size=max(1, user_lens[i] // 2)).tolist()
                final[s] += reply_len
        if free_between and t + 1 < turns:
            for s in ids:
                ops.append(("free", s))
        else:
            live += ids
    need = sum(-(-L // B) for L in final.values())
    nb = pool if pool is not None else max(1, int(math.ceil(1.2 * need)))
    free_order = rng.permutation(nb).astype(np.int32)
    return Workload(name=name or f"shared prefix: {n_requests} requests x (system {system_len} + user), "
                                 f"{turns} turn(s), H={H}, D={D}, B={B}, {dtype}",
                    num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=sigma, num_blocks=nb,
                    free_order=free_order, ops=ops, seed=seed, final_lens=final)


def decode_steps(prompt_lens, steps: int, *, H=2, D=128, B=16, dtype="f16", sigma=1.0, seed=9,
                 drop_every: int = 0, small_first: int = 0, name=None) -> Workload:
    """Prompts, then ``steps`` decode steps, each followed by attention over the batch.
    With ``drop_every`` > 0, every ``drop_every``-th sequence sits out every other step,
    so the batch (and its size) changes from step to step.  With ``small_first`` > 0,
    only the first ``small_first`` sequences take part in the first half of the steps."""
    prompt_lens = [int(x) for x in prompt_lens]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    final = [L + steps for L in prompt_lens]
    nb = _pool_size(final, B)
    free_order = rng.permutation(nb).astype(np.int32)
    ops = [("add", s, L) for s, L in enumerate(prompt_lens)]
    counts = [0] * len(prompt_lens)
    for k in range(steps):
        seqs = tuple(s for s in range(len(prompt_lens))
                     if not (drop_every and s % drop_every == 0 and k % 2 == 1)
                     and not (small_first and k < steps // 2 and s >= small_first))
        for s in seqs:
            counts[s] += 1
        ops.append(("step", seqs))
        ops.append(("attend", seqs))
    return Workload(name=name or f"decode steps: {len(prompt_lens)} seqs x {steps} steps, H={H}, D={D}, B={B}, "
                                 f"{dtype}",
                    num_heads=H, head_dim=D, block_size=B, dtype=dtype, sigma=sigma, num_blocks=nb,
                    free_order=free_order, ops=ops, seed=seed,
                    final_lens={s: L + c for s, (L, c) in enumerate(zip(prompt_lens, counts))})


def custom(lengths, *, H=2, D=128, B=16, dtype="f16", sigma=1.0, seed=7, shuffle=True,
           pool=None, free_order=None, name=None) -> Workload:
    """Decode batch with explicit final context lengths (edge cases, sweeps)."""
    return _decode_batch(name or f"custom L={list(lengths)[:6]}..., H={H}, D={D}, B={B}, {dtype}",
                         lengths, H, D, B, dtype, sigma, seed, shuffle=shuffle, pool=pool,
                         free_order=free_order)
