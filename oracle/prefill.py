"""Multi-query (prefill) attention through block tables (oracle, test only).

Sources:
* "PagedAttention, clearly explained": the cache keeps each token's keys and
  values so that later tokens can attend over the prompt without recomputing
  it; the attention kernel gathers them through the block table.
* katajob Q&A, "What the KV cache is": every earlier token's key and value
  must be available to the attention of the next token; "The paging idea": a
  sequence starts with just enough blocks for its prompt.
* foundry page on paged block allocation, "Failure modes": reused blocks and
  freshly prefilled ones meet inside one attention reduction (prefill runs over
  cached prefixes).

Reading (the pages describe no prefill kernel): a prefill chunk of sequence s
is its last n_s logical positions ctx_s - n_s .. ctx_s - 1, whose keys and
values are already in the pool (written by the slot write, like a decode
step's token).  The query at position p attends to positions 0 .. p of the
same sequence (itself and everything before it, the autoregressive order).
With n_s = 1 this is decode attention.  Grouped-query mapping as in decode:
query head j reads KV head j // (Hq / N_kv).

The plain definition, in fp64: logits = Q K^T * scale over the gathered K,
positions after p masked out, softmax with the row maximum subtracted, times V.
A matrix product serves as the dot-product step.
"""
from __future__ import annotations

import numpy as np

from .attention import gather_sequence, head_scale


def causal_mask(first_pos: int, n_queries: int, ctx: int) -> np.ndarray:
    """[n_queries, ctx] boolean: query i (position first_pos + i) sees
    positions 0 .. first_pos + i."""
    pos = np.arange(ctx)[None, :]
    qpos = first_pos + np.arange(n_queries)[:, None]
    return pos <= qpos


def paged_attention_prefill(q: np.ndarray, pool, tables, context_lens, query_start,
                            softmax_scale: float, k_scale: float = 1.0,
                            v_scale: float = 1.0, seqs=None) -> np.ndarray:
    """Prefill attention of a batch.

    q: fp64 [total_q, Hq, D], the queries of sequence s in rows
    query_start[s] .. query_start[s + 1] - 1 (positions ctx_s - n_s ..).
    pool: a ``PoolModel``; tables: per sequence its block ids in logical order;
    context_lens: [B] (chunk included).  ``seqs`` restricts the work to some
    sequences (the other rows stay NaN).  Returns fp64 [total_q, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    total_q, hq, d = q.shape
    n_kv = pool.num_kv_heads
    group = hq // n_kv
    qs = np.asarray(query_start, dtype=np.int64)
    out = np.full((total_q, hq, d), np.nan, dtype=np.float64)
    rows = range(len(context_lens)) if seqs is None else seqs
    for s in rows:
        ctx = int(context_lens[s])
        r0, r1 = int(qs[s]), int(qs[s + 1])
        n = r1 - r0
        if n == 0:
            continue
        if n > ctx:
            raise ValueError(f"sequence {s}: {n} queries but context {ctx}")
        mask = causal_mask(ctx - n, n, ctx)
        for h in range(n_kv):
            k = gather_sequence(pool.k, tables[s], ctx, h, pool.block_size, pool.kv_dtype,
                                head_scale(k_scale, h))
            v = gather_sequence(pool.v, tables[s], ctx, h, pool.block_size, pool.kv_dtype,
                                head_scale(v_scale, h))
            for j in range(h * group, (h + 1) * group):
                logits = (q[r0:r1, j] @ k.T) * softmax_scale
                logits = np.where(mask, logits, -np.inf)
                w = np.exp(logits - logits.max(axis=1, keepdims=True))
                out[r0:r1, j] = (w @ v) / w.sum(axis=1, keepdims=True)
    return out
