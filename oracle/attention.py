"""Single-token decode attention through block tables (oracle, test only).

Sources:
* "PagedAttention, clearly explained": at each decode step the attention
  kernel reads the block table and gathers keys and values from whichever
  physical blocks they landed in.
* foundry page on paged block allocation, "Concept": attention needs its keys
  and values ordered by position, not adjacent in memory; the output is a
  weighted sum over positions.  "In and out": relocation is not
  transformation; the output is the ordinary attention output.
* katajob Q&A, "The paging idea": each sequence owns an ordered list of
  physical block ids for its logical positions.

So the oracle is the plain definition: for sequence s and logical position p
the key is K_pool[table[s][p // T], h, p % T, :]; the output of query head j
is softmax(q_j . K^T * scale) V over positions 0 .. ctx_s - 1, computed in
fp64 with the maximum subtracted before the exponential.

Readings where the pages are silent:
* Grouped-query attention maps query head j to KV head j // (Hq / N_kv).
* A context length of zero yields a zero output.
* The context length counts the token written in this step.
* An E4M3 cache is read as e4m3 * scale with one scale per tensor, or one
  per KV head (k_scale, v_scale given as arrays [N_kv]; the pages fix only
  the one-byte element size, so the per-head variant is the same decoding
  with KV head h's own scale).
"""
from __future__ import annotations

import numpy as np

from .pool import bits_to_f64


def gather_sequence(cache: dict, table, ctx: int, kv_head: int, block_size: int,
                    kv_dtype: str, scale: float = 1.0) -> np.ndarray:
    """Contiguous fp64 [ctx, head_dim] K (or V) of one sequence and KV head,
    position by position through the block table."""
    p = np.arange(ctx)
    block_of_p = np.asarray(table, dtype=np.int64)[p // block_size]
    offset_of_p = p % block_size
    blocks, which = np.unique(block_of_p, return_inverse=True)
    tiles = np.stack([cache[int(b)][kv_head] for b in blocks])  # [n_blocks, T, D]
    return bits_to_f64(tiles[which, offset_of_p], kv_dtype, scale)


def head_scale(scale, h: int) -> float:
    """The E4M3 scale that KV head h is read with: the number itself for a
    per-tensor scale, element h of a per-head array."""
    a = np.asarray(scale)
    return float(a.reshape(-1)[h]) if a.ndim else float(a)


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V for one query vector, fp64."""
    logits = (k @ q) * scale
    w = np.exp(logits - logits.max())
    return (w @ v) / w.sum()


def paged_attention_decode(q: np.ndarray, pool, tables, context_lens, softmax_scale: float,
                           k_scale: float = 1.0, v_scale: float = 1.0,
                           seqs=None) -> np.ndarray:
    """Decode attention of a batch.

    q: fp64 [B, Hq, D]; pool: a ``PoolModel`` (blocks of raw storage bits);
    tables: per sequence a list of block ids (logical block order);
    context_lens: [B].  ``seqs`` restricts the work to some batch rows (the
    other rows of the result stay NaN).  Returns fp64 [B, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    b_, hq, d = q.shape
    n_kv = pool.num_kv_heads
    group = hq // n_kv
    out = np.full((b_, hq, d), np.nan, dtype=np.float64)
    rows = range(b_) if seqs is None else seqs
    for s in rows:
        ctx = int(context_lens[s])
        for h in range(n_kv):
            if ctx == 0:
                out[s, h * group:(h + 1) * group] = 0.0
                continue
            k = gather_sequence(pool.k, tables[s], ctx, h, pool.block_size, pool.kv_dtype,
                                head_scale(k_scale, h))
            v = gather_sequence(pool.v, tables[s], ctx, h, pool.block_size, pool.kv_dtype,
                                head_scale(v_scale, h))
            for j in range(h * group, (h + 1) * group):
                out[s, j] = softmax_attention(q[s, j], k, v, softmax_scale)
    return out
