"""Block allocator with prefix caching (oracle, test infrastructure only).

Sources:
* foundry page on paged block allocation, "The knobs": with prefix caching the
  engine hashes each filled block so that unrelated requests share physical
  blocks, not just forks of one sequence; prefix hashes are computed per
  block, so sharing is as coarse as the block size.
* same page, "Failure modes": sharing is block-granular: with block size 32 a
  shared 1,000-token prefix reuses at most 992 tokens, and any divergence
  inside a block loses that whole block.
* katajob Q&A, "Sharing, the second dividend": if the tokens match, the blocks
  holding their KV state are reused across requests and that part of prefill
  is skipped.

Readings where the pages are silent:
* A full block whose token ids are known is published under the exact key
  (entry of the previous block of its sequence, its block_size token ids);
  entry 0 stands for "no previous block", published entries are numbered 1,
  2, ... in publication order.  When the key is already published (another
  block holds the same content) the sequence refers to that entry and keeps
  its own block unpublished.
* A new request takes, block by block from its first, the published blocks
  whose keys match its prompt, at most (n_tokens - 1) // block_size of them:
  at least one prompt token is always computed (its output is the reason the
  prompt runs).
* A published block whose count drops to zero stays published and joins the
  reusable list; finishing a sequence adds its published blocks last block
  first.  Blocks are taken from the free stack first and, when it is empty,
  from the front of the reusable list (eviction: the entry is dropped).
* Ids of a sequence's positions are kept only while all earlier ids are
  known; a block is published only if its whole prefix chain is.
"""
from __future__ import annotations

from .allocator import AllocError, BlockAllocator


class PrefixCachingAllocator(BlockAllocator):
    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        super().__init__(num_blocks, block_size, initial_free_order)
        self.next_entry = 1
        self.key_to_entry: dict[tuple, int] = {}
        self.entry_block: dict[int, int] = {}
        self.entry_key: dict[int, tuple] = {}
        self.block_entry = [-1] * self.num_blocks
        self.reuse: list[int] = []          # front = first to be evicted
        self.tokens: dict[int, list[int]] = {}
        self.chain: dict[int, list[int]] = {}
        self.hit_tokens = 0
        self.evictions = 0

    # ---------------------------------------------------------------- queries
    def num_free(self) -> int:
        return len(self.free) + len(self.reuse)

    def reusable(self) -> list[int]:
        return list(self.reuse)

    def stats(self):
        return (len(self.entry_block), len(self.reuse), self.hit_tokens, self.evictions)

    # --------------------------------------------------------------- internals
    def _take(self) -> int:
        if self.free:
            return self.free.pop()
        b = self.reuse.pop(0)
        self._drop_entry(b)
        self.evictions += 1
        return b

    def _drop_entry(self, b: int):
        e = self.block_entry[b]
        if e >= 0:
            del self.key_to_entry[self.entry_key.pop(e)]
            del self.entry_block[e]
            self.block_entry[b] = -1

    def _publish(self, seq: int):
        t = self.block_size
        tab, toks, ch = self.tables[seq], self.tokens[seq], self.chain[seq]
        for i in range(len(ch), self.lens[seq] // t):
            parent = 0 if i == 0 else ch[i - 1]
            if parent < 0 or len(toks) < (i + 1) * t:
                ch.append(-1)
                continue
            key = (parent, tuple(toks[i * t:(i + 1) * t]))
            if key in self.key_to_entry:
                ch.append(self.key_to_entry[key])
                continue
            b = tab[i]
            if self.block_entry[b] >= 0:    # a fork sibling published this very block
                ch.append(self.block_entry[b])
                continue
            e = self.next_entry
            self.next_entry += 1
            self.key_to_entry[key] = e
            self.entry_key[e] = key
            self.entry_block[e] = b
            self.block_entry[b] = e
            ch.append(e)

    # -------------------------------------------------------------- mutations
    def create(self, seq: int):
        super().create(seq)
        self.tokens[seq] = []
        self.chain[seq] = []

    def create_cached(self, seq: int, token_ids) -> int:
        """A new sequence holding the cached blocks that match its prompt;
        returns the number of prompt tokens it holds."""
        self.create(seq)
        ids = [int(x) for x in token_ids]
        t = self.block_size
        tab, ch = self.tables[seq], self.chain[seq]
        for i in range(max(0, (len(ids) - 1) // t)):
            key = (0 if i == 0 else ch[-1], tuple(ids[i * t:(i + 1) * t]))
            e = self.key_to_entry.get(key)
            if e is None:
                break
            b = self.entry_block[e]
            if b in self.reuse:
                self.reuse.remove(b)
            self.refcount[b] += 1
            tab.append(b)
            ch.append(e)
        self.lens[seq] = len(tab) * t
        self.tokens[seq] = ids[:self.lens[seq]]
        self.hit_tokens += self.lens[seq]
        return self.lens[seq]

    def append(self, seq: int, n_new: int, token_ids=None):
        self._need(seq)
        if n_new < 0:
            raise AllocError("INVALID_ARG", "negative token count")
        need, cow = self._blocks_needed(seq, n_new)
        if need > self.num_free():
            raise AllocError("OUT_OF_BLOCKS", f"need {need}, {self.num_free()} free")
        t = self.block_size
        tab = self.tables[seq]
        start = self.lens[seq]
        slots, pairs = [], []
        for p in range(start, start + n_new):
            if p % t == 0:
                b = self._take()
                self.refcount[b] = 1
                tab.append(b)
            elif p == start and cow:
                src = tab[p // t]
                dst = self._take()
                self.refcount[dst] = 1
                self.refcount[src] -= 1
                tab[p // t] = dst
                pairs.append((src, dst))
            slots.append(tab[p // t] * t + p % t)
        if token_ids is not None and len(self.tokens[seq]) == start:
            self.tokens[seq] += [int(x) for x in token_ids]
        self.lens[seq] = start + n_new
        self._publish(seq)
        return slots, pairs

    def fork(self, parent: int, child: int):
        super().fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])
        self.chain[child] = list(self.chain[parent])

    def free_seq(self, seq: int):
        self._need(seq)
        tab = self.tables[seq]
        for b in reversed(tab):
            if self.block_entry[b] >= 0:
                self.refcount[b] -= 1
                if self.refcount[b] == 0:
                    self.reuse.append(b)
        for b in tab:
            if self.block_entry[b] < 0:
                self.refcount[b] -= 1
                if self.refcount[b] == 0:
                    self.free.append(b)
        del self.tables[seq]
        del self.lens[seq]
        del self.tokens[seq]
        del self.chain[seq]
