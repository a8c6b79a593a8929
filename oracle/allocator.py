"""Block allocator model (oracle, test infrastructure only).

Sources:
* foundry page on paged block allocation, "In and out": the free pool is a
  stack of physical indices into one pre-allocated tensor; blocks are
  allocated on demand, one per block_size tokens, each index appended to the
  sequence's block table; a reference count is incremented when a block is
  shared with a fork.
* same page, "Concept": forking copies the table rather than the memory, and a
  block is copied only when one branch writes into it (copy-on-write).
* "PagedAttention, clearly explained": a block is assigned only when the
  previous one fills; when a request finishes its block numbers go straight
  back to the pool.
* "PagedAttention Memory Management", "Complex Topologies and Memory Sharing":
  shared prompt blocks carry a reference count equal to the number of
  sequences mapping them.

Readings where the pages are silent (each one needed for bit-exact tables):
* The free stack is LIFO.  The initial order is given top first; by default
  block 0 is on top, then 1, 2, ...
* Freeing a sequence walks its table in logical order, decrements each
  block's count and pushes the block when the count reaches zero, so the
  sequence's last block ends on top.
* Copy-on-write happens when a token is written into a partly filled last
  block whose count is above one: a fresh block is popped, the pair
  (src, dst) is reported, the source count drops by one and this sequence's
  table entry is replaced.  A full shared block is never copied; the next
  token opens a new block.
* Every call is all-or-nothing: on error nothing changes.
"""
from __future__ import annotations

import copy


class AllocError(Exception):
    """Raised with ``code`` one of: INVALID_ARG, OUT_OF_BLOCKS, UNKNOWN_SEQ."""

    def __init__(self, code: str, msg: str = ""):
        super().__init__(f"{code}: {msg}")
        self.code = code


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise AllocError("INVALID_ARG", "pool and block size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if initial_free_order is None:
            order = list(range(self.num_blocks))
        else:
            order = [int(b) for b in initial_free_order]
            if sorted(order) != list(range(self.num_blocks)):
                raise AllocError("INVALID_ARG", "initial order must be a permutation of the pool")
        # Python list used as a stack: the top is the end of the list.
        self.free = list(reversed(order))
        self.refcount = [0] * self.num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    # ---------------------------------------------------------------- queries
    def num_free(self) -> int:
        return len(self.free)

    def free_stack_top_first(self) -> list[int]:
        return list(reversed(self.free))

    def table(self, seq: int) -> list[int]:
        self._need(seq)
        return list(self.tables[seq])

    def context_len(self, seq: int) -> int:
        self._need(seq)
        return self.lens[seq]

    def block_refcount(self, block: int) -> int:
        if not 0 <= block < self.num_blocks:
            raise AllocError("INVALID_ARG", "block id out of range")
        return self.refcount[block]

    def _need(self, seq: int):
        if seq not in self.tables:
            raise AllocError("UNKNOWN_SEQ", str(seq))

    # -------------------------------------------------------------- mutations
    def create(self, seq: int):
        if seq in self.tables:
            raise AllocError("INVALID_ARG", f"sequence {seq} exists")
        self.tables[seq] = []
        self.lens[seq] = 0

    def _blocks_needed(self, seq: int, n_new: int) -> tuple[int, bool]:
        """Blocks one append of n_new tokens pops, and whether it copies."""
        length, tab, t = self.lens[seq], self.tables[seq], self.block_size
        cow = n_new > 0 and length % t != 0 and self.refcount[tab[length // t]] > 1
        opened = sum(1 for p in range(length, length + n_new) if p % t == 0)
        return opened + (1 if cow else 0), cow

    def append(self, seq: int, n_new: int):
        """Reserve slots for n_new tokens of one sequence.

        Returns (slots, cow_pairs): the physical slot of each new token,
        block * block_size + offset, and the (src, dst) block copies that must
        run before the tokens are written.
        """
        self._need(seq)
        if n_new < 0:
            raise AllocError("INVALID_ARG", "negative token count")
        need, cow = self._blocks_needed(seq, n_new)
        if need > len(self.free):
            raise AllocError("OUT_OF_BLOCKS", f"need {need}, {len(self.free)} free")
        t = self.block_size
        tab = self.tables[seq]
        start = self.lens[seq]
        slots, pairs = [], []
        for p in range(start, start + n_new):
            if p % t == 0:
                b = self.free.pop()
                self.refcount[b] = 1
                tab.append(b)
            elif p == start and cow:
                src = tab[p // t]
                dst = self.free.pop()
                self.refcount[dst] = 1
                self.refcount[src] -= 1
                tab[p // t] = dst
                pairs.append((src, dst))
            slots.append(tab[p // t] * t + p % t)
        self.lens[seq] = start + n_new
        return slots, pairs

    def append_batch(self, seqs, n_new: int = 1):
        """One append per sequence, in the given order; all-or-nothing over
        the whole batch.  Returns (slots, cow_pairs) concatenated in order."""
        trial = copy.deepcopy(self)
        all_slots, all_pairs = [], []
        for s in seqs:
            sl, pr = trial.append(s, n_new)
            all_slots += sl
            all_pairs += pr
        self.__dict__.update(trial.__dict__)
        return all_slots, all_pairs

    def fork(self, parent: int, child: int):
        """The child maps the parent's blocks; every shared block gains a count."""
        self._need(parent)
        if child in self.tables:
            raise AllocError("INVALID_ARG", f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free_seq(self, seq: int):
        """Finish a sequence: its blocks whose count reaches zero go back on
        the stack, in logical order."""
        self._need(seq)
        for b in self.tables[seq]:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.tables[seq]
        del self.lens[seq]

    # ------------------------------------------------------------- accounting
    def padded_tables(self, seqs, width: int | None = None, pad: int = -1):
        """Block tables of ``seqs`` as rows of equal width, padded with ``pad``."""
        rows = [self.tables[s] for s in seqs]
        w = max((len(r) for r in rows), default=0) if width is None else width
        return [r + [pad] * (w - len(r)) for r in rows]
