"""Preemption by recompute and admission with a free-block watermark (oracle,
test infrastructure only).

Sources:
* foundry page on paged block allocation, "The knobs": when the pool cannot
  satisfy a running sequence the engine preempts it, drops its blocks and
  re-prefills it later; swapping is gone, recompute is the only mode.
* same page, "Effect": when the free-block pool runs dry the scheduler
  preempts running sequences rather than failing them, and under sustained
  pressure a request can be preempted and restarted several times.
* same page, "Failure modes": repeated preemption under steady load means the
  free-block watermark is hit constantly.
* katajob Q&A, "Operational consequences": under overload the pool still
  fills; preempted sequences have their blocks freed and their state is
  recomputed on readmission.

Readings where the pages are silent:
* In a decode step the batch order is the priority order.  When a sequence
  cannot get its block, the lowest-priority sequence still running (the last
  one of the batch not yet preempted, possibly the one being served) is
  preempted: its blocks are freed as when it finishes, and it leaves the
  pool; a preempted sequence gets no token in this step.
* Admission of a new sequence (its whole prompt at once) requires that at
  least `watermark` blocks stay free after it; decode appends of running
  sequences are not held back by the watermark.
"""
from __future__ import annotations

from .allocator import AllocError


def append_batch_preempt(alloc, seqs):
    """One token per sequence of ``seqs`` (priority order).

    Returns (slots, cow_pairs, preempted): slots[i] is -1 for a preempted
    sequence; preempted lists the preempted ids in the order they were
    preempted.
    """
    seqs = [int(s) for s in seqs]
    for s in seqs:
        if s not in alloc.tables:
            raise AllocError("UNKNOWN_SEQ", str(s))
    if len(set(seqs)) != len(seqs):
        raise AllocError("INVALID_ARG", "a sequence appears twice in the batch")
    running = list(range(len(seqs)))       # indices still running, priority order
    slots = [-1] * len(seqs)
    pairs, preempted = [], []
    for i, s in enumerate(seqs):
        if i not in running:
            continue
        while True:
            need, _ = alloc._blocks_needed(s, 1)
            if need <= alloc.num_free():
                sl, pr = alloc.append(s, 1)
                slots[i] = sl[0]
                pairs += pr
                break
            victim = running.pop()          # the lowest priority still running
            alloc.free_seq(seqs[victim])
            preempted.append(seqs[victim])
            if victim == i:
                break
    return slots, pairs, preempted


def admit(alloc, seq: int, n_tokens: int, watermark: int):
    """Create ``seq`` with ``n_tokens`` tokens if at least ``watermark``
    blocks stay free afterwards; returns its slots."""
    if n_tokens < 0 or watermark < 0:
        raise AllocError("INVALID_ARG", "negative size")
    if seq in alloc.tables:
        raise AllocError("INVALID_ARG", f"sequence {seq} exists")
    need = -(-n_tokens // alloc.block_size)
    if need + watermark > alloc.num_free():
        raise AllocError("OUT_OF_BLOCKS", f"need {need} + watermark {watermark}, {alloc.num_free()} free")
    alloc.create(seq)
    return alloc.append(seq, n_tokens)[0]
