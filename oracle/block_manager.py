"""Block tables, free list, reference counts and copy-on-write, on the host.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rules, as the pages state them:

* [note] 关键设计 2 ("Block table 与按需分配"), [guide] 03: each sequence has a
  list of logical blocks; each records its physical block id and how many of
  its token slots are filled.  Prefill takes just enough blocks for the
  prompt; each decode token goes to the last block, and a new physical block
  is taken only once the last one is full, so at most one block per sequence
  is partly filled (0 <= tail waste < B tokens).
* [lecture] PagedAttention 原理: the worked example -- a 7-token prompt with B=4
  fills logical block 0 (4 tokens) and logical block 1 (3 tokens + 1 free
  slot); "fathers" fills block 1; "brought" goes to a newly taken block 2.
* [note] 关键设计 3 ("共享、引用计数与写时复制"), [guide] 04 step 4, [lecture]
  Parallel Sampling 场景: a physical block shared by several logical blocks
  carries a reference count.  A sequence about to write into a shared block
  (count > 1) takes a new block, has the old content copied into it, lowers
  the old block's count by one and points its logical block at the copy; a
  block whose count is 1 is written in place.
* [guide] 04 (shared prefix): the provider stores a prefix's blocks ahead of
  time; a request maps its first logical blocks onto them, the last one
  marked copy-on-write.
* [lecture] Beam Search 场景 / [note] 失败案例 4: sharing is driven by three
  actions, fork, append and free; freeing returns blocks whose count drops
  to zero.

Readings where the pages are silent or garbled (each test pins one):

* The order in which a full last block and a shared last block are checked:
  a full block is never written again, so fullness is checked first and a
  full shared block needs no copy.  After taking a new block for a full last
  block, the token is written to the new block (the page's listing keeps
  using the old block's fill counter; the prose says the new token goes to
  the new block).
* Newly taken blocks start with reference count 1.
* The free list is a FIFO over a caller-given order of physical ids: taking
  pops the front, a freed block is pushed at the back (in logical order when
  a whole sequence is freed).
* A registered prefix holds one reference on each of its blocks, so a request
  that writes into a partly filled last prefix block always copies it.
* Running out of blocks raises ``MemoryError`` and changes nothing.
* slot = physical id * B + row.
* Swapping ([lecture] 调度和抢占; [guide] 05): a preempted group of sequences
  moves, whole, to a second manager that tracks a host pool, and back the same
  way.  The group must hold every reference to its blocks (its samples or beams
  share blocks with each other, not with sequences left behind, and not with a
  registered prefix); each distinct block gets one block on the other side, in
  order of first appearance (sequences in the given order, each in logical
  order), and carries its reference count; the old blocks return to their free
  list in the same order.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Sequence, Tuple


class LogicalBlock:
    __slots__ = ("physical", "filled")

    def __init__(self, physical: int, filled: int):
        self.physical = physical
        self.filled = filled


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.B = block_size
        self.num_blocks = num_blocks
        self.free_list = deque(order)
        self.ref = [0] * num_blocks
        self.seqs: Dict[int, List[LogicalBlock]] = {}
        self.prefixes: Dict[int, List[LogicalBlock]] = {}
        self.cow_copies = 0
        self.prefix_seqs = 0          # sequences added on a registered prefix
        self.prefix_blocks = 0        # block references they took from prefixes
        self.groups_out = self.blocks_out = self.groups_in = self.blocks_in = 0

    # -- physical blocks -------------------------------------------------
    def _take(self) -> int:
        block = self.free_list.popleft()
        self.ref[block] = 1
        return block

    def _release(self, block: int) -> None:
        self.ref[block] -= 1
        if self.ref[block] < 0:
            raise RuntimeError(f"reference count of block {block} went negative")
        if self.ref[block] == 0:
            self.free_list.append(block)

    def _need(self, n: int) -> None:
        if n > len(self.free_list):
            raise MemoryError(f"need {n} free blocks, have {len(self.free_list)}")

    def _fresh_blocks(self, num_tokens: int) -> List[LogicalBlock]:
        n = -(-num_tokens // self.B)
        self._need(n)
        blocks = []
        for j in range(n):
            blocks.append(LogicalBlock(self._take(), min(self.B, num_tokens - j * self.B)))
        return blocks

    def _slots(self, blocks: List[LogicalBlock]) -> List[int]:
        return [b.physical * self.B + r for b in blocks for r in range(b.filled)]

    # -- sequences -------------------------------------------------------
    def add_seq(self, seq_id: int, prompt_len: int) -> List[int]:
        """Prefill: take ceil(prompt_len / B) blocks; return the prompt tokens' slots."""
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        if prompt_len <= 0:
            raise ValueError("prompt_len must be positive")
        blocks = self._fresh_blocks(prompt_len)
        self.seqs[seq_id] = blocks
        return self._slots(blocks)

    def fork(self, parent: int, child: int) -> None:
        """The child maps every logical block onto the parent's physical block."""
        if child in self.seqs:
            raise ValueError(f"sequence {child} exists")
        src = self.seqs[parent]
        for b in src:
            self.ref[b.physical] += 1
        self.seqs[child] = [LogicalBlock(b.physical, b.filled) for b in src]

    def append_slot(self, seq_id: int) -> Tuple[int, int, int]:
        """Find the slot of the sequence's next token.

        Returns (slot, copy_src, copy_dst); copy_src = copy_dst = -1 unless the
        write needed a copy of a shared block first.
        """
        blocks = self.seqs[seq_id]
        last = blocks[-1]
        src = dst = -1
        if last.filled == self.B:
            # full: the token starts a new logical block on a newly taken physical block
            self._need(1)
            last = LogicalBlock(self._take(), 0)
            blocks.append(last)
        elif self.ref[last.physical] > 1:
            # shared and partly filled: copy it, move this sequence onto the copy
            self._need(1)
            new = self._take()
            src, dst = last.physical, new
            self.ref[last.physical] -= 1
            last.physical = new
            self.cow_copies += 1
        slot = last.physical * self.B + last.filled
        last.filled += 1
        return slot, src, dst

    def extend(self, seq_id: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """n appends to one sequence, all or nothing ([guide] 04: the prompt phase places a
        request's whole task input at once).  Returns (slots in order, copies made).

        The blocks the n appends will take are counted first by walking the same decisions
        append_slot makes (full last block -> a new block; shared partly filled last block -> a
        copy, after which the block is private), so a short free list raises MemoryError before
        anything changes.
        """
        if n < 0:
            raise ValueError("n must be non-negative")
        last = self.seqs[seq_id][-1]
        filled, shared, need = last.filled, self.ref[last.physical] > 1, 0
        for _ in range(n):
            if filled == self.B:
                need, filled, shared = need + 1, 0, False
            elif shared:
                need, shared = need + 1, False
            filled += 1
        self._need(need)
        slots, copies = [], []
        for _ in range(n):
            slot, src, dst = self.append_slot(seq_id)
            slots.append(slot)
            if src >= 0:
                copies.append((src, dst))
        return slots, copies

    def free(self, seq_id: int) -> None:
        for b in self.seqs.pop(seq_id):
            self._release(b.physical)

    # -- provider-stored prefixes -----------------------------------------
    def register_prefix(self, prefix_id: int, length: int) -> List[int]:
        """Take and hold blocks for a prefix; return its tokens' slots (to be filled once)."""
        if prefix_id in self.prefixes:
            raise ValueError(f"prefix {prefix_id} exists")
        if length <= 0:
            raise ValueError("length must be positive")
        blocks = self._fresh_blocks(length)
        self.prefixes[prefix_id] = blocks
        return self._slots(blocks)

    def add_seq_with_prefix(self, seq_id: int, prefix_id: int,
                            suffix_len: int = 0) -> Tuple[List[int], List[Tuple[int, int]]]:
        """A request whose first logical blocks are the prefix's physical blocks ([guide] 04 steps
        2 and 4), followed by ``suffix_len`` tokens of its own (the task input).  Returns the
        suffix tokens' slots and the copies made (at most one: a partly filled last prefix block
        is shared with the prefix).  All or nothing: MemoryError leaves the state unchanged."""
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        if suffix_len < 0:
            raise ValueError("suffix_len must be non-negative")
        src = self.prefixes[prefix_id]
        for b in src:
            self.ref[b.physical] += 1
        self.seqs[seq_id] = [LogicalBlock(b.physical, b.filled) for b in src]
        try:
            out = self.extend(seq_id, suffix_len)
        except MemoryError:
            for b in self.seqs.pop(seq_id):
                self.ref[b.physical] -= 1
            raise
        self.prefix_seqs += 1
        self.prefix_blocks += len(src)
        return out

    def drop_prefix(self, prefix_id: int) -> None:
        for b in self.prefixes.pop(prefix_id):
            self._release(b.physical)

    # -- views -------------------------------------------------------------
    def block_table(self, seq_id: int) -> Tuple[List[int], int]:
        blocks = self.seqs[seq_id]
        return [b.physical for b in blocks], sum(b.filled for b in blocks)

    def filled(self, seq_id: int) -> List[int]:
        return [b.filled for b in self.seqs[seq_id]]

    def ref_count(self, block: int) -> int:
        return self.ref[block]

    def num_free(self) -> int:
        return len(self.free_list)

    def ref_histogram(self, cap: int = 8) -> List[int]:
        """Blocks per reference count r < cap - 1; the last entry counts every larger count."""
        hist = [0] * cap
        for r in self.ref:
            hist[min(r, cap - 1)] += 1
        return hist

    def counters(self) -> Dict[str, int]:
        return {"cow_copies": self.cow_copies, "prefix_seqs": self.prefix_seqs, "prefix_blocks": self.prefix_blocks,
                "groups_out": self.groups_out, "blocks_out": self.blocks_out, "groups_in": self.groups_in,
                "blocks_in": self.blocks_in}

    def tail_waste_tokens(self) -> int:
        """Sum over sequences of the unfilled slots of their blocks."""
        return sum(self.B * len(bl) - sum(b.filled for b in bl) for bl in self.seqs.values())

    # -- beam search ---------------------------------------------------------
    def beam_step(self, parents, children, retire):
        """One beam-search step ([lecture] Beam Search 场景; [guide] 04, beam search).

        Each new candidate children[i] shares every block of parents[i] (a fork);
        then the retired candidates (the previous beam, dropped or not) are freed,
        so blocks no candidate still holds return to the free list -- back up the
        tree to, but not including, blocks the survivors share; then every new
        candidate appends its token, copying a shared partly filled last block
        (the one-block copy of beam search).  All or nothing: on MemoryError
        nothing has changed.
        Returns [(slot, copy_src, copy_dst)] in the order of ``children``.
        """
        import copy
        if len(parents) != len(children):
            raise ValueError("parents and children differ in length")
        if len(set(children)) != len(children) or any(c in self.seqs for c in children):
            raise ValueError("children must be new, distinct ids")
        if any(p not in self.seqs for p in parents) or any(r not in self.seqs for r in retire):
            raise KeyError("unknown parent or retired sequence")
        if len(set(retire)) != len(retire):
            raise ValueError("a sequence is retired twice")
        trial = copy.deepcopy(self)
        trial._beam_step_unchecked(parents, children, retire)       # raises MemoryError if short
        return self._beam_step_unchecked(parents, children, retire)

    def _beam_step_unchecked(self, parents, children, retire):
        for p, c in zip(parents, children):
            self.fork(p, c)
        for r in retire:
            self.free(r)
        return [self.append_slot(c) for c in children]


# -- swapping ------------------------------------------------------------------
def swap(src: BlockManager, dst: BlockManager, seq_ids: Sequence[int]) -> List[Tuple[int, int]]:
    """Move the sequences ``seq_ids`` (a whole group) from ``src`` to ``dst``.

    Returns the block moves [(src block, dst block)] the caller makes with
    swap_blocks before the sequences run again on ``dst``'s pool.  All or
    nothing: a bad id, a block the group does not hold alone, or a short free
    list on ``dst`` (MemoryError) changes neither manager.
    """
    ids = [int(s) for s in seq_ids]
    if src is dst or src.B != dst.B:
        raise ValueError("swap needs two managers with the same block size")
    if len(set(ids)) != len(ids):
        raise ValueError("a sequence is listed twice")
    if any(s not in src.seqs for s in ids):
        raise KeyError("unknown sequence")
    if any(s in dst.seqs for s in ids):
        raise ValueError("a sequence already exists on the destination")
    held: Dict[int, int] = {}                 # block -> references the group holds
    order: List[int] = []                     # distinct blocks, first appearance first
    for s in ids:
        for b in src.seqs[s]:
            if b.physical not in held:
                held[b.physical] = 0
                order.append(b.physical)
            held[b.physical] += 1
    for b in order:
        if held[b] != src.ref[b]:
            raise ValueError(f"block {b} is also held outside the group")
    dst._need(len(order))
    moved = {}
    for b in order:
        nb = dst._take()
        dst.ref[nb] = src.ref[b]
        moved[b] = nb
    for s in ids:
        dst.seqs[s] = [LogicalBlock(moved[b.physical], b.filled) for b in src.seqs.pop(s)]
    for b in order:
        src.ref[b] = 0
        src.free_list.append(b)
    if ids:
        src.groups_out += 1
        dst.groups_in += 1
    src.blocks_out += len(order)
    dst.blocks_in += len(order)
    return [(b, moved[b]) for b in order]
