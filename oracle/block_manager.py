"""Oracle block manager: free-list paging with reference counts and copy-on-write.

Follows "PagedAttention: Virtual Memory Guide for LLM Inference":
  * "The Mathematics of Block Translation": token i of a sequence lives in logical
    block floor(i/B) at offset i mod B; the block table maps the logical block to a
    physical frame.
  * "Key Architectural Mechanics / 1. Demand Paging": a new token t goes to offset
    t mod B of the current frame; when t mod B == 0 one free frame is popped and
    appended to the table.
  * "Key Architectural Mechanics / 2. Zero-Copy Branching via Copy-on-Write": a fork
    shares every frame (reference count + 1); writing into a shared frame first
    moves the writer onto a private copy of that one frame.
  * "Reference Implementation": free frames leave from the FRONT of the free list
    and return to its BACK when their count reaches zero; releasing a frame whose
    count is already zero does nothing; a sequence that is not known is ignored on
    free.
and "Solving the LLM Memory Wall" ("Implementation", BlockManager.allocate): a
prompt's blocks are granted all-or-nothing -- the free count is checked before any
frame leaves the list.

Readings where the pages leave a step open:
  * the block boundary test comes before looking at the tail frame, so an empty
    prompt (no frames yet) takes its first frame on the first append;
  * copy-on-write allocates the private frame first, then drops one reference from
    the shared frame, then puts the private frame in the tail position; the data
    copy (shared -> private) is reported to the caller;
  * several sequences appended in one step are served in the order given;
  * a step is all-or-nothing: if any append in it cannot get a frame, no state
    changes.
"""

from __future__ import annotations

import copy
from collections import deque

DOUBLE_FREE = "double-free"


class OutOfBlocks(Exception):
    pass


class UnknownSequence(KeyError):
    pass


class SequenceExists(KeyError):
    pass


class OracleBlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_list: deque[int] = deque(order)
        self.refs: list[int] = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    # -- frame pool ----------------------------------------------------------------
    def _take_frame(self) -> int:
        if len(self.free_list) == 0:
            raise OutOfBlocks("no free physical block")
        frame = self.free_list.popleft()
        self.refs[frame] = 1
        return frame

    def _drop_ref(self, frame: int) -> None:
        if self.refs[frame] <= 0:          # already free: nothing to release
            return
        self.refs[frame] -= 1
        if self.refs[frame] == 0:
            self.free_list.append(frame)

    # -- translation -----------------------------------------------------------------
    def slot(self, seq: int, i: int) -> int:
        """Flat slot index of token i: frame * B + offset."""
        table = self.tables[seq]
        logical, offset = divmod(i, self.block_size)
        return table[logical] * self.block_size + offset

    # -- sequence operations ---------------------------------------------------------------
    def add_seq(self, seq: int, num_tokens: int) -> list[int]:
        """Frames for a prompt of num_tokens, granted all-or-nothing. Returns its slots."""
        if seq in self.tables:
            raise SequenceExists(seq)
        if num_tokens < 0:
            raise ValueError("negative prompt length")
        frames_needed = -(-num_tokens // self.block_size)
        if frames_needed > len(self.free_list):
            raise OutOfBlocks(f"prompt needs {frames_needed} blocks, {len(self.free_list)} free")
        self.tables[seq] = [self._take_frame() for _ in range(frames_needed)]
        self.lens[seq] = num_tokens
        return [self.slot(seq, i) for i in range(num_tokens)]

    def append(self, seq: int):
        """One new token: returns (slot, copy) where copy is (src, dst) or None."""
        if seq not in self.tables:
            raise UnknownSequence(seq)
        t = self.lens[seq]
        table = self.tables[seq]
        copy_pair = None
        if t % self.block_size == 0:
            table.append(self._take_frame())
        else:
            shared = table[-1]
            if self.refs[shared] > 1:
                private = self._take_frame()
                self._drop_ref(shared)
                table[-1] = private
                copy_pair = (shared, private)
        self.lens[seq] = t + 1
        return self.slot(seq, t), copy_pair

    def step(self, seqs):
        """One decode step over seqs in order; all-or-nothing on OutOfBlocks.

        Returns (slots, copies) with copies in issue order.
        """
        saved = (copy.copy(self.free_list), list(self.refs),
                 {s: list(t) for s, t in self.tables.items()}, dict(self.lens))
        slots, copies = [], []
        try:
            for s in seqs:
                slot, pair = self.append(s)
                slots.append(slot)
                if pair is not None:
                    copies.append(pair)
        except (OutOfBlocks, UnknownSequence):
            self.free_list, self.refs, self.tables, self.lens = saved
            raise
        return slots, copies

    def extend(self, seq: int, n: int):
        """n new tokens for one sequence (a prompt chunk), all-or-nothing.

        Each token follows the single-token rule in turn.  Returns (slots, copies)."""
        if seq not in self.tables:
            raise UnknownSequence(seq)
        return self.step([seq] * int(n))

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.tables:
            raise UnknownSequence(parent)
        if child in self.tables:
            raise SequenceExists(child)
        for frame in self.tables[parent]:
            self.refs[frame] += 1
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]

    def free(self, seq: int):
        """Release a finished sequence; an unknown sequence is a no-op (returns DOUBLE_FREE)."""
        if seq not in self.tables:
            return DOUBLE_FREE
        for frame in self.tables[seq]:
            self._drop_ref(frame)
        del self.tables[seq]
        del self.lens[seq]
        return None

    # -- views ---------------------------------------------------------------------------
    @property
    def free_count(self) -> int:
        return len(self.free_list)

    def fill_levels(self, seq: int):
        """Tokens held by each frame of seq's table, in table order."""
        L, B = self.lens[seq], self.block_size
        return [min(B, L - j * B) for j in range(len(self.tables[seq]))]

    def _cached_free_frames(self) -> int:
        return 0  # no prefix cache in the plain manager

    def usage(self) -> dict:
        """Memory accounting of the pool.

        "PagedAttention: Virtual Memory Guide for LLM Inference", "The Solution": frames
        come on demand, so only the unfilled slots of a sequence's last frame are wasted
        (fewer than B per sequence); "2. Zero-Copy Branching via Copy-on-Write": forked
        sequences hold their shared frames once.  "Solving the LLM Memory Wall",
        "Performance Analysis": slots allocated against tokens held.
        """
        B = self.block_size
        filled = {}  # frame -> the most slots any sequence holding it has filled
        entries = tokens = worst = 0
        for s, table in self.tables.items():
            L = self.lens[s]
            entries += len(table)
            tokens += L
            worst = max(worst, len(table) * B - L)
            for j, frame in enumerate(table):
                held = min(B, max(0, L - j * B))
                filled[frame] = max(filled.get(frame, 0), held)
        in_use = [f for f in range(self.num_blocks) if self.refs[f] > 0]
        return {
            "num_seqs": len(self.tables),
            "frames_total": self.num_blocks,
            "frames_in_use": len(in_use),
            "frames_cached": self._cached_free_frames(),
            "table_entries": entries,
            "tokens_logical": tokens,
            "slots_filled": sum(filled.get(f, 0) for f in in_use),
            "max_seq_waste": worst,
        }

    def snapshot(self):
        return {
            "tables": {s: list(t) for s, t in self.tables.items()},
            "lens": dict(self.lens),
            "free": list(self.free_list),
            "refs": list(self.refs),
        }
