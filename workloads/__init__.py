"""Seeded synthetic inputs for the paged KV-cache decode workloads.

This module is the only code shared by the CPU oracle (``oracle/``) and the CUDA
product path (``paged_kv_cache_137_gb300/``).  It draws random numbers and casts
them to storage dtypes; it holds none of the method's arithmetic (no block
tables, no slots, no attention).  Every draw comes from its own numpy PCG64
stream keyed by (config seed, purpose, index), so a test can regenerate the
inputs of one sequence without drawing the whole workload.

The five workloads follow the synthetic configurations the method is measured
on (decode of one new token per sequence over a pool of fixed-size blocks):

* ``tiny_fp32``        1 layer, 4 seqs, 4 q heads = 4 KV heads, head_dim 64,
                       block 16, pool 64 blocks, ctx ~ U[1,128], fp32.
* ``qwen_gqa_bf16``    28 q heads / 4 KV heads, head_dim 128, block 16, pool
                       8,500 blocks, 64 seqs, ctx ~ U[256,4096], bf16.
* ``prefix_fork_bf16`` 32 q / 8 KV heads, head_dim 128, block 16, 256 seqs
                       sharing a 1,024-token prefix, private tails ~ U[1,512],
                       25% of sequences forked mid-block (copy-on-write), bf16.
* ``long_mha_bf16``    32 q = 32 KV heads, head_dim 128, block 32, 8 seqs,
                       ctx ~ U[16384,32768], every 97th key scaled by 8, bf16,
                       512-token split-K partitions.
* ``fp8_churn``        64 q / 8 KV heads, head_dim 128, block 16, 512 seqs,
                       ctx log-uniform on [64,8192], E4M3 KV with one scale per
                       tensor, pool 65,536 blocks scrambled by 10k alloc/free
                       churn operations.

Ranges are integer and inclusive; values are N(0,1) drawn in fp32 and rounded
to the storage dtype with PyTorch's round-to-nearest-even cast.  A workload
with ``head_gain_log2`` g > 0 multiplies KV head h's keys and values by
2^(-g h) in fp32 before the cast (heads of very different magnitude, the case
per-head FP8 scales are for).
"""
from __future__ import annotations

import math
import functools
from dataclasses import dataclass, replace

import numpy as np
import torch

__all__ = [
    "q_for_chunk", "chunk_lens",
    "Workload", "CONFIGS", "get", "scaled",
    "rng", "context_lens", "free_order", "churn_ops", "q_for_seq", "kv_for_seq",
    "prefix_kv", "fork_layout", "fp8_scales", "kv_amax", "TORCH_DTYPES",
    "head_gains", "kv_amax_heads", "fp8_head_scales",
]

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Purpose keys of the independent random streams.
_CTX, _ORDER, _CHURN, _Q, _K, _V, _PREFIX_K, _PREFIX_V, _TAIL, _PREFILL_Q = range(10)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    kv_dtype: str              # "f32" | "f16" | "bf16" | "e4m3"
    q_dtype: str               # "f32" | "f16" | "bf16"
    ctx_range: tuple = (1, 1)  # inclusive
    ctx_dist: str = "uniform"  # "uniform" | "loguniform" | "prefix_fork"
    num_layers: int = 1
    prefix_len: int = 0
    tail_range: tuple = (0, 0)
    fork_fraction: float = 0.0
    spike_every: int = 0       # every n-th logical key (1-based) is scaled
    spike_scale: float = 1.0
    partition_tokens: int = 0  # split-K partition size, 0 = library default
    churn: int = 0             # alloc/free operations applied before the workload
    shuffled_pool: bool = True
    prefill_chunk: int = 0     # > 0: a prefill workload, chunks of the last positions
    head_gain_log2: float = 0.0  # KV head h's K and V multiplied by 2^(-head_gain_log2 * h)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def kv_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else (4 if self.kv_dtype == "f32" else 2)

    @property
    def src_dtype(self) -> str:
        """dtype of the new K/V handed to the slot write (the q dtype)."""
        return self.q_dtype


CONFIGS = {
    "tiny_fp32": Workload(
        name="tiny_fp32", seed=1371, num_seqs=4, num_q_heads=4, num_kv_heads=4,
        head_dim=64, block_size=16, num_blocks=64, kv_dtype="f32", q_dtype="f32",
        ctx_range=(1, 128)),
    "qwen_gqa_bf16": Workload(
        name="qwen_gqa_bf16", seed=1372, num_seqs=64, num_q_heads=28, num_kv_heads=4,
        head_dim=128, block_size=16, num_blocks=8500, kv_dtype="bf16", q_dtype="bf16",
        ctx_range=(256, 4096)),
    "prefix_fork_bf16": Workload(
        name="prefix_fork_bf16", seed=1373, num_seqs=256, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, num_blocks=8192, kv_dtype="bf16", q_dtype="bf16",
        ctx_dist="prefix_fork", prefix_len=1024, tail_range=(1, 512), fork_fraction=0.25),
    "long_mha_bf16": Workload(
        name="long_mha_bf16", seed=1374, num_seqs=8, num_q_heads=32, num_kv_heads=32,
        head_dim=128, block_size=32, num_blocks=8192, kv_dtype="bf16", q_dtype="bf16",
        ctx_range=(16384, 32768), spike_every=97, spike_scale=8.0, partition_tokens=512),
    "fp8_churn": Workload(
        name="fp8_churn", seed=1375, num_seqs=512, num_q_heads=64, num_kv_heads=8,
        head_dim=128, block_size=16, num_blocks=65536, kv_dtype="e4m3", q_dtype="bf16",
        ctx_range=(64, 8192), ctx_dist="loguniform", churn=10000),
    # chunked prefill on the Qwen-shaped layer: each sequence's last 512
    # positions are the chunk, attending to its cached prefix and causally
    # within the chunk
    "qwen_prefill_bf16": Workload(
        name="qwen_prefill_bf16", seed=1376, num_seqs=16, num_q_heads=28, num_kv_heads=4,
        head_dim=128, block_size=16, num_blocks=4500, kv_dtype="bf16", q_dtype="bf16",
        ctx_range=(1024, 4096), prefill_chunk=512),
}


def get(name: str) -> Workload:
    return CONFIGS[name]


def scaled(w: Workload, **overrides) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return replace(w, **overrides)


def rng(w: Workload, purpose: int, index: int = 0, attempt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, purpose, index, attempt])))


def _cast(x32: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(TORCH_DTYPES[dtype])


def _blocks(n: int, t: int) -> int:
    return -(-n // t)


def context_lens(w: Workload) -> np.ndarray:
    """Attended context length per sequence (the new token included).

    For ``uniform`` and ``loguniform`` draws the lengths are redrawn (attempt
    1, 2, ...) until the whole batch fits the pool; the attempt that was
    accepted is recorded in ``last_attempt``.  ``prefix_fork`` lengths are
    prefix + tail (see :func:`fork_layout`).
    """
    if w.ctx_dist == "prefix_fork":
        return fork_layout(w)["ctx"]
    lo, hi = w.ctx_range
    for attempt in range(1000):
        g = rng(w, _CTX, 0, attempt)
        if w.ctx_dist == "uniform":
            ctx = g.integers(lo, hi, size=w.num_seqs, endpoint=True)
        elif w.ctx_dist == "loguniform":
            u = g.uniform(math.log(lo), math.log(hi), size=w.num_seqs)
            ctx = np.clip(np.floor(np.exp(u)), lo, hi)
        else:
            raise ValueError(w.ctx_dist)
        ctx = ctx.astype(np.int64)
        if sum(_blocks(int(c), w.block_size) for c in ctx) <= w.num_blocks:
            context_lens.last_attempt = attempt
            return ctx
    raise RuntimeError("no context-length draw fits the pool")


context_lens.last_attempt = 0


def free_order(w: Workload) -> np.ndarray:
    """Initial free-stack order, top first: a random permutation of the pool
    (or 0, 1, 2, ... when the pool is not shuffled)."""
    if not w.shuffled_pool:
        return np.arange(w.num_blocks, dtype=np.int32)
    return rng(w, _ORDER).permutation(w.num_blocks).astype(np.int32)


def churn_ops(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Random numbers for the allocate/free churn: per operation a coin in
    [0,1) (allocate when < 0.5) and a pick in [0,1) that selects which live
    block to free as floor(pick * live_count)."""
    g = rng(w, _CHURN)
    coin = g.random(w.churn)
    pick = g.random(w.churn)
    return coin, pick


def q_for_seq(w: Workload, seq: int) -> torch.Tensor:
    """q of one sequence, [num_q_heads, head_dim] in the q dtype."""
    x = rng(w, _Q, seq).standard_normal((w.num_q_heads, w.head_dim), dtype=np.float32)
    return _cast(x, w.q_dtype)


def q_for_chunk(w: Workload, seq: int, n_tokens: int) -> torch.Tensor:
    """Queries of a prefill chunk of ``n_tokens`` tokens of one sequence,
    [n_tokens, num_q_heads, head_dim] in the q dtype (their own stream, so they
    do not depend on the decode queries)."""
    x = rng(w, _PREFILL_Q, seq).standard_normal((n_tokens, w.num_q_heads, w.head_dim),
                                                 dtype=np.float32)
    return _cast(x, w.q_dtype)


def chunk_lens(w: Workload, ctx, chunk: int) -> np.ndarray:
    """Prefill chunk lengths: the last min(ctx, chunk) positions of each
    sequence are its chunk (a sequence shorter than the chunk is a whole
    prompt)."""
    return np.minimum(np.asarray(ctx, dtype=np.int64), chunk)


def kv_for_seq(w: Workload, seq: int, n_tokens: int, first_pos: int = 0,
               stream_index: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """K and V of ``n_tokens`` tokens at logical positions first_pos.. of one
    sequence, each [n_tokens, num_kv_heads, head_dim] in the source dtype.

    The draws of one sequence come from its own stream, so that the K/V of
    positions [a, b) do not depend on how the range is cut into calls: the
    stream is advanced past ``first_pos`` tokens first.  Keys at logical
    positions p with (p + 1) % spike_every == 0 are multiplied by spike_scale
    in fp32 before the cast.
    """
    idx = seq if stream_index is None else stream_index
    per_tok = w.num_kv_heads * w.head_dim
    out = []
    for purpose in (_K, _V):
        g = rng(w, purpose, idx)
        if first_pos:
            _ = g.standard_normal(first_pos * per_tok, dtype=np.float32)
        x = g.standard_normal((n_tokens, w.num_kv_heads, w.head_dim), dtype=np.float32)
        if purpose == _K and w.spike_every:
            pos = np.arange(first_pos, first_pos + n_tokens)
            hit = (pos + 1) % w.spike_every == 0
            x[hit] *= np.float32(w.spike_scale)
        if w.head_gain_log2:
            x *= head_gains(w)[None, :, None]
        out.append(_cast(x, w.src_dtype))
    return out[0], out[1]


def head_gains(w: Workload) -> np.ndarray:
    """fp32 [num_kv_heads]: the factor 2^(-head_gain_log2 * h) of KV head h."""
    h = np.arange(w.num_kv_heads, dtype=np.float64)
    return np.exp2(-w.head_gain_log2 * h).astype(np.float32)


def prefix_kv(w: Workload) -> tuple[torch.Tensor, torch.Tensor]:
    """K/V of the shared prefix of the prefix-fork workload."""
    per = (w.prefix_len, w.num_kv_heads, w.head_dim)
    k = rng(w, _PREFIX_K).standard_normal(per, dtype=np.float32)
    v = rng(w, _PREFIX_V).standard_normal(per, dtype=np.float32)
    if w.head_gain_log2:
        k *= head_gains(w)[None, :, None]
        v *= head_gains(w)[None, :, None]
    return _cast(k, w.src_dtype), _cast(v, w.src_dtype)


def fork_layout(w: Workload) -> dict:
    """Structure of the prefix-fork workload.

    ``num_parents = num_seqs * (1 - fork_fraction)`` parents share the prefix
    and each owns a private tail drawn from ``tail_range``; a parent's prior
    length before the decode step is prefix + tail - 1.  The first
    ``num_children`` parents whose prior length is not a multiple of the block
    size (a fork in the middle of a block) each get one child.  The batch
    order is children first, then parents; ``ctx`` is in batch order, and a
    child attends the same length as its parent.  The prefix is whole blocks
    (its last block full), so every parent's tail starts in a block of its
    own and only the decode step copies blocks.
    """
    if w.prefix_len % w.block_size:
        raise ValueError(f"prefix_len {w.prefix_len} is not a multiple of block_size {w.block_size}")
    n_children = int(round(w.num_seqs * w.fork_fraction))
    n_parents = w.num_seqs - n_children
    lo, hi = w.tail_range
    for attempt in range(1000):
        tails = rng(w, _TAIL, 0, attempt).integers(lo, hi, size=n_parents, endpoint=True)
        prior = w.prefix_len + tails - 1
        mid = np.nonzero(prior % w.block_size != 0)[0]
        if len(mid) >= n_children:
            parent_of_child = mid[:n_children].astype(np.int64)
            ctx_parents = (w.prefix_len + tails).astype(np.int64)
            ctx = np.concatenate([ctx_parents[parent_of_child], ctx_parents])
            return {"tails": tails.astype(np.int64), "parent_of_child": parent_of_child,
                    "num_parents": n_parents, "num_children": n_children, "ctx": ctx}
    raise RuntimeError("could not draw enough mid-block forks")


def fp8_scales(amax_k, amax_v) -> dict:
    """E4M3 scales from the absolute maxima of the K (V) values: scale =
    amax / 448 in fp32 and the reciprocal the slot write multiplies by,
    inv = fp32(1 / scale).  448 is the largest finite E4M3 value.  Numbers
    give per-tensor scales (floats); arrays [N_kv] give per-KV-head scales
    (float32 arrays)."""
    out = {}
    for name, a in (("k", amax_k), ("v", amax_v)):
        s = np.asarray(a, dtype=np.float32) / np.float32(448.0)
        inv = np.float32(1.0) / s
        scalar = np.ndim(a) == 0
        out[name + "_scale"] = float(s) if scalar else s.astype(np.float32)
        out[name + "_inv_scale"] = float(inv) if scalar else inv.astype(np.float32)
    return out


@functools.lru_cache(maxsize=8)
def kv_amax_heads(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Largest |K| and |V| of each KV head over every token of every sequence
    of a workload (positions 0 .. ctx - 1, in the source dtype): float64
    arrays [num_kv_heads], the statistic per-head E4M3 scales come from."""
    if w.ctx_dist == "prefix_fork":
        raise NotImplementedError("scales from maxima are defined for independent sequences")
    ak = np.zeros(w.num_kv_heads)
    av = np.zeros(w.num_kv_heads)
    for s, c in enumerate(context_lens(w)):
        k, v = kv_for_seq(w, s, int(c))
        ak = np.maximum(ak, k.float().abs().amax(dim=(0, 2)).double().numpy())
        av = np.maximum(av, v.float().abs().amax(dim=(0, 2)).double().numpy())
    return ak, av


def kv_amax(w: Workload) -> tuple[float, float]:
    """Largest |K| and |V| over every token of every sequence of a workload,
    the statistic the per-tensor E4M3 scales are computed from."""
    ak, av = kv_amax_heads(w)
    return float(ak.max()), float(av.max())


def fp8_head_scales(w: Workload) -> dict:
    """Per-KV-head E4M3 scales of a workload (fp8_scales of the per-head maxima)."""
    return fp8_scales(*kv_amax_heads(w))
