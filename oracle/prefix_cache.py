"""Oracle block manager with prefix caching -- TEST INFRASTRUCTURE ONLY.

"PagedAttention: Virtual Memory Guide for LLM Inference", "2. Native Synergy with
RadixAttention and Prompt Caching": once a block is filled it is immutable, so a
later request whose token prefix is identical maps that part of its block table
onto the same physical frames instead of recomputing it (the comparison table
calls it chunk-level prefix reuse).

Readings taken where the page leaves the mechanics open:
  * Only full blocks are shared.  A full block is identified exactly by its
    content prefix: the node of the block before it plus its own B token ids, a
    trie of blocks (no hashing, so no false matches).  Each registered block is a
    node with a fresh id that is never reused; a key names the parent by that id,
    so a child of an evicted block can no longer be reached.
  * Admission looks up the prompt's leading full blocks in order and stops at the
    first miss; it never maps the last token (at least one query of a prompt is
    always computed), i.e. only blocks that end at or before token L-2 can hit.
    A hit frame gets one more reference; if it had none it leaves the free list.
  * Blocks are registered when they become full with known tokens: at admission
    (the prompt's full blocks past the hits) and when appends with token ids fill
    a block.  If the key is already registered (the same content computed twice),
    the existing node stands for the block's content and this frame stays
    unregistered.  An append without a token id leaves its block unregistered
    (and every later block of that sequence); a sequence admitted without token
    ids (and its forks) never registers anything.
  * A freed frame keeps its contents and its registration and goes to the back of
    the free list like any other; it is evicted (its node removed) only when the
    free list hands it out again.  Frames are therefore evicted least recently
    freed first, with the base manager's free-list order unchanged.
  * Admission is all-or-nothing: hits that sit in the free list count against the
    frames available for the rest of the prompt.
"""

from __future__ import annotations

import copy

from .block_manager import OracleBlockManager, OutOfBlocks, SequenceExists, UnknownSequence


class OraclePrefixBlockManager(OracleBlockManager):
    ROOT = 0

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        super().__init__(num_blocks, block_size, free_order)
        self.node_of_key: dict[tuple, int] = {}      # (parent node id, block tokens) -> node id
        self.node_frame: dict[int, int] = {}         # node id -> frame holding the block
        self.node_key: dict[int, tuple] = {}         # node id -> its key
        self.frame_node: list[int] = [0] * num_blocks  # frame -> node id registered on it (0: none)
        self.next_node = 1
        self.tokens: dict[int, list] = {}            # seq -> token ids (None entries: unknown)
        self.nodes: dict[int, list] = {}             # seq -> node id per block (0: none)
        self.tracked: set[int] = set()               # sequences admitted with token ids

    # -- frame pool: a frame handed out again loses its registration -----------------------
    def _take_frame(self) -> int:
        frame = super()._take_frame()
        node = self.frame_node[frame]
        if node:
            self._evict(node)
        return frame

    def _evict(self, node: int) -> None:
        frame = self.node_frame.pop(node)
        key = self.node_key.pop(node)
        del self.node_of_key[key]
        self.frame_node[frame] = 0

    def _key(self, parent: int, toks) -> tuple:
        return (parent, tuple(toks))

    def _hit_limit(self, L: int) -> int:
        """Tokens a lookup may cover: never the last one of the prompt."""
        return L - 1

    def _revive(self, frame: int) -> None:
        if self.refs[frame] == 0:
            self.free_list.remove(frame)
        self.refs[frame] += 1

    def _register(self, seq: int, block: int) -> None:
        """Block `block` of seq has just become full with known tokens."""
        B = self.block_size
        toks = self.tokens[seq][block * B:(block + 1) * B]
        nodes = self.nodes[seq]
        if seq not in self.tracked:
            return
        parent = self.ROOT if block == 0 else nodes[block - 1]
        if any(t is None for t in toks) or parent == 0 and block > 0:
            nodes[block] = 0
            return
        key = self._key(parent, toks)
        existing = self.node_of_key.get(key)
        if existing is not None:                      # same content already registered
            nodes[block] = existing
            return
        node = self.next_node
        self.next_node += 1
        frame = self.tables[seq][block]
        self.node_of_key[key] = node
        self.node_frame[node] = frame
        self.node_key[node] = key
        self.frame_node[frame] = node
        nodes[block] = node

    # -- sequences ------------------------------------------------------------------------
    def add_seq(self, seq: int, num_tokens: int) -> list[int]:
        slots = super().add_seq(seq, num_tokens)
        self.tokens[seq] = [None] * num_tokens
        self.nodes[seq] = [0] * len(self.tables[seq])
        return slots

    def add_seq_cached(self, seq: int, tokens):
        """Admit a prompt given by its token ids.  Returns (n_cached, slots) where the
        first n_cached tokens are already in the cache and slots are those of the
        remaining tokens (to be written by the caller)."""
        if seq in self.tables:
            raise SequenceExists(seq)
        tokens = [int(t) for t in tokens]
        B, L = self.block_size, len(tokens)
        hits = []          # (node, frame) of leading blocks found in the cache
        parent = self.ROOT
        while (len(hits) + 1) * B <= self._hit_limit(L):
            i = len(hits)
            node = self.node_of_key.get(self._key(parent, tokens[i * B:(i + 1) * B]))
            if node is None:
                break
            hits.append((node, self.node_frame[node]))
            parent = node
        n_blocks = -(-L // B)
        new_needed = n_blocks - len(hits)
        available = len(self.free_list) - sum(1 for _, f in hits if self.refs[f] == 0)
        if new_needed > available:
            raise OutOfBlocks(f"prompt needs {new_needed} new blocks, {available} available")
        for _, f in hits:                             # revive or share
            self._revive(f)
        table = [f for _, f in hits]
        self.tables[seq] = table
        self.lens[seq] = L
        self.tokens[seq] = list(tokens)
        self.nodes[seq] = [n for n, _ in hits]
        self.tracked.add(seq)
        for i in range(len(hits), n_blocks):
            table.append(self._take_frame())
            self.nodes[seq].append(0)
            if (i + 1) * B <= L:
                self._register(seq, i)
        n_cached = len(hits) * B
        return n_cached, [self.slot(seq, i) for i in range(n_cached, L)]

    def append(self, seq: int, token=None):
        if seq not in self.tables:
            raise UnknownSequence(seq)
        t = self.lens[seq]
        slot, pair = super().append(seq)
        self.tokens[seq].append(None if token is None else int(token))
        nodes = self.nodes[seq]
        if len(nodes) < len(self.tables[seq]):
            nodes.append(0)
        if (t + 1) % self.block_size == 0:
            self._register(seq, t // self.block_size)
        return slot, pair

    def _save(self):
        return (copy.copy(self.free_list), list(self.refs), {s: list(t) for s, t in self.tables.items()},
                dict(self.lens), dict(self.node_of_key), dict(self.node_frame), dict(self.node_key),
                list(self.frame_node), self.next_node, {s: list(t) for s, t in self.tokens.items()},
                {s: list(n) for s, n in self.nodes.items()}, set(self.tracked))

    def _restore(self, saved):
        (self.free_list, self.refs, self.tables, self.lens, self.node_of_key, self.node_frame, self.node_key,
         self.frame_node, self.next_node, self.tokens, self.nodes, self.tracked) = saved

    def step(self, seqs, tokens=None):
        """One decode step (tokens[i] is the id appended to seqs[i], or None)."""
        saved = self._save()
        slots, copies = [], []
        try:
            for i, s in enumerate(seqs):
                slot, pair = self.append(s, None if tokens is None else tokens[i])
                slots.append(slot)
                if pair is not None:
                    copies.append(pair)
        except (OutOfBlocks, UnknownSequence):
            self._restore(saved)
            raise
        return slots, copies

    def extend(self, seq: int, n: int, tokens=None):
        if seq not in self.tables:
            raise UnknownSequence(seq)
        return self.step([seq] * int(n), tokens)

    def fork(self, parent: int, child: int) -> None:
        super().fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])
        self.nodes[child] = list(self.nodes[parent])
        if parent in self.tracked:
            self.tracked.add(child)

    def free(self, seq: int):
        r = super().free(seq)
        if r is None:
            del self.tokens[seq]
            del self.nodes[seq]
            self.tracked.discard(seq)
        return r

    # -- views --------------------------------------------------------------------------
    def _cached_free_frames(self) -> int:
        free = set(self.free_list)
        return sum(1 for f, n in enumerate(self.frame_node) if n and f in free)

    def cached_frames(self) -> list[int]:
        """1 for each frame that holds a registered block, else 0."""
        return [1 if n else 0 for n in self.frame_node]

    def snapshot(self):
        snap = super().snapshot()
        snap["cached"] = self.cached_frames()
        return snap
