"""The synthetic decode workloads, built with the oracle's own pieces (test only).

Each workload is: an allocator over a pool (optionally scrambled by churn), a
prefill of every sequence's prior tokens, then one decode step that appends
one token per sequence, copies shared blocks that are about to be written
(copy-on-write), writes the new K/V and runs decode attention.

Readings (the pages describe the mechanism, not these workloads):
* Prefill appends a sequence's ctx - 1 prior tokens in one call, sequences in
  batch order; the decode step appends one token per sequence in batch order.
* Churn: each operation allocates one block as a fresh one-block sequence when
  its coin is below 0.5 and a block is free (or nothing is live), otherwise it
  finishes the live one-block sequence at index floor(pick * live_count) of the
  live list (kept in allocation order).  All churn sequences are finished
  afterwards, in live-list order.
* Prefix fork: parent 0 prefills the prefix, the other parents fork it, every
  parent then prefills its private tail; each child forks its parent.  The
  batch is the children followed by the parents.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import workloads as W

from .allocator import BlockAllocator
from .pool import PoolModel

CHURN_SEQ_BASE = 1 << 40

POISON = {"f32": 0xFFFFFFFF, "f16": 0xFFFF, "bf16": 0xFFFF, "e4m3": 0xFF}


def torch_bits(t) -> np.ndarray:
    """Raw storage bits of a CPU tensor (16- or 32-bit float)."""
    import torch
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).numpy().view(np.uint32)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class Scenario:
    w: W.Workload
    alloc: BlockAllocator
    pool: PoolModel
    seq_ids: list                  # batch row -> sequence id
    ctx: np.ndarray                # [B] attended lengths
    q_bits: np.ndarray             # [B, Hq, D] raw bits of q (q dtype)
    step_slots: list               # [B] slot of each new token
    cow_pairs: list                # (src, dst) copies run before the step's write
    scales: dict = field(default_factory=dict)

    @property
    def tables(self):
        return [self.alloc.table(s) for s in self.seq_ids]

    def q_f64(self):
        from .pool import bits_to_f64
        return bits_to_f64(self.q_bits, self.w.q_dtype)


def apply_churn(alloc: BlockAllocator, coin, pick, block_size: int):
    live, next_id = [], CHURN_SEQ_BASE
    for c, p in zip(coin, pick):
        if (c < 0.5 and alloc.num_free() > 0) or not live:
            alloc.create(next_id)
            alloc.append(next_id, block_size)
            live.append(next_id)
            next_id += 1
        else:
            alloc.free_seq(live.pop(int(p * len(live))))
    for s in live:
        alloc.free_seq(s)


def build(w: W.Workload, write_seqs=None, scales: dict | None = None) -> Scenario:
    """Build a workload.  ``write_seqs`` (batch rows) limits which sequences'
    K/V are stored in the pool model (all when None); the allocator always runs
    the whole workload.  ``scales`` are the per-tensor E4M3 scales (required
    for an E4M3 cache)."""
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    if w.churn:
        apply_churn(alloc, *W.churn_ops(w), w.block_size)
    pool = PoolModel(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, w.kv_dtype,
                     POISON[w.kv_dtype])
    scales = dict(scales or {})
    kinv = scales.get("k_inv_scale", 1.0)
    vinv = scales.get("v_inv_scale", 1.0)
    if w.kv_dtype == "e4m3" and "k_inv_scale" not in scales:
        raise ValueError("an E4M3 cache needs its scales")

    def write(slots, k, v):
        pool.write(torch_bits(k), torch_bits(v), w.src_dtype, slots, kinv, vinv)

    ctx = W.context_lens(w)
    if w.ctx_dist == "prefix_fork":
        lay = W.fork_layout(w)
        n_par, n_ch = lay["num_parents"], lay["num_children"]
        seq_ids = [n_par + c for c in range(n_ch)] + list(range(n_par))
        row_of = {s: r for r, s in enumerate(seq_ids)}
        want = set(range(len(seq_ids)) if write_seqs is None else write_seqs)
        alloc.create(0)
        slots, _ = alloc.append(0, w.prefix_len)
        pk, pv = W.prefix_kv(w)
        write(slots, pk, pv)
        for p in range(1, n_par):
            alloc.fork(0, p)
        for p in range(n_par):
            n_tail = int(lay["tails"][p]) - 1
            slots, _ = alloc.append(p, n_tail)
            if row_of[p] in want or any(int(lay["parent_of_child"][c]) == p and row_of[n_par + c] in want
                                        for c in range(n_ch)):
                k, v = W.kv_for_seq(w, p, n_tail, first_pos=w.prefix_len)
                write(slots, k, v)
        for c in range(n_ch):
            alloc.fork(int(lay["parent_of_child"][c]), n_par + c)
    else:
        seq_ids = list(range(w.num_seqs))
        want = set(range(len(seq_ids)) if write_seqs is None else write_seqs)
        for r, s in enumerate(seq_ids):
            alloc.create(s)
            slots, _ = alloc.append(s, int(ctx[r]) - 1)
            if r in want:
                k, v = W.kv_for_seq(w, s, int(ctx[r]) - 1)
                write(slots, k, v)

    # decode step: append one token per sequence, copy-on-write, write, attend
    step_slots, cow_pairs = alloc.append_batch(seq_ids, 1)
    pool.copy_blocks(cow_pairs)
    for r, s in enumerate(seq_ids):
        if r in want:
            k, v = W.kv_for_seq(w, s, 1, first_pos=int(ctx[r]) - 1)
            write([step_slots[r]], k, v)
    q_bits = np.stack([torch_bits(W.q_for_seq(w, s)) for s in seq_ids])
    return Scenario(w=w, alloc=alloc, pool=pool, seq_ids=seq_ids, ctx=np.asarray(ctx),
                    q_bits=q_bits, step_slots=step_slots, cow_pairs=cow_pairs, scales=scales)
