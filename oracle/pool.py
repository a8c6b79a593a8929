"""The physical K/V pool: slot writes and block copies (oracle, test only).

Sources:
* "PagedAttention, clearly explained": the pool of numbered, equally sized
  physical blocks is the only KV memory; each block holds the keys and values
  of block_size consecutive tokens.
* foundry page on paged block allocation, "In and out": one large
  pre-allocated tensor per layer; the step writes the new tokens' K/V.
* same page, "Concept": a shared block is copied only when a branch writes
  into it (copy-on-write).

Readings (the pages fix no in-block layout):
* Per layer, K and V are separate tensors laid out [num_blocks, N_kv,
  block_size, head_dim]; a block id indexes the same slot range in every
  layer's tensors.
* Slot s is block s // block_size, offset s % block_size.  A negative slot
  means "write nothing" for that token.
* An FP8 (E4M3) cache stores the byte of fp32(x * inv_scale); 16- and 32-bit
  caches store the input's bits unchanged.  The inverse scale is one number
  per tensor, or one per KV head (an array of N_kv values): head h of every
  token is then multiplied by its own inv_scale[h].
* A block copy copies the raw bytes of K and V of every layer.

Storage is kept as raw bit patterns (uint16 for f16/bf16, uint32 for f32,
uint8 for E4M3) in a dict from block id to an array [N_kv, block_size,
head_dim]; a block that was never written does not exist, so reading it is an
error.  ``dense`` lays the blocks out as the full pool with a fill pattern.
"""
from __future__ import annotations

import numpy as np

from . import e4m3

STORAGE = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}


def bits_to_f64(bits: np.ndarray, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Values held by raw storage bits, as fp64 (E4M3 times its scale)."""
    bits = np.asarray(bits)
    if dtype == "f32":
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "e4m3":
        return e4m3.decode(bits) * np.float64(np.float32(scale))
    raise ValueError(dtype)


def f32_of_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values of 16/32-bit source bits (exact upcast)."""
    return bits_to_f64(bits, dtype).astype(np.float32)


class PoolModel:
    """One layer's K and V pools as sparse blocks of raw storage bits."""

    def __init__(self, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
                 kv_dtype: str, fill: int):
        self.num_blocks = num_blocks
        self.num_kv_heads = num_kv_heads
        self.block_size = block_size
        self.head_dim = head_dim
        self.kv_dtype = kv_dtype
        self.fill = fill
        self.k: dict[int, np.ndarray] = {}
        self.v: dict[int, np.ndarray] = {}

    def _fresh(self):
        shape = (self.num_kv_heads, self.block_size, self.head_dim)
        return np.full(shape, self.fill, dtype=STORAGE[self.kv_dtype])

    def write(self, k_bits: np.ndarray, v_bits: np.ndarray, src_dtype: str, slots,
              k_inv_scale=1.0, v_inv_scale=1.0):
        """Store token i's K/V [N_kv, head_dim] at slot slots[i].  The inverse
        scales are numbers (per tensor) or arrays [N_kv] (per KV head)."""
        slots = [int(s) for s in slots]
        for cache, src, inv in ((self.k, k_bits, k_inv_scale), (self.v, v_bits, v_inv_scale)):
            if self.kv_dtype == "e4m3":
                inv = np.asarray(inv, dtype=np.float32)
                if inv.ndim:                  # per KV head: axis 1 of [tokens, N_kv, D]
                    if inv.shape != (self.num_kv_heads,):
                        raise ValueError("per-head scales need one value per KV head")
                    inv = inv.reshape(1, -1, 1)
                stored = e4m3.quantize_fp32(f32_of_bits(src, src_dtype), inv)
            else:
                if src_dtype != self.kv_dtype:
                    raise ValueError("16/32-bit caches store the input dtype")
                stored = np.asarray(src).astype(STORAGE[self.kv_dtype])
            for i, s in enumerate(slots):
                if s < 0:
                    continue
                b, off = divmod(s, self.block_size)
                if b >= self.num_blocks:
                    raise IndexError("slot outside the pool")
                if b not in cache:
                    cache[b] = self._fresh()
                cache[b][:, off, :] = stored[i]

    def copy_blocks(self, pairs):
        """Block copy: dst takes src's bytes (K and V), pairs in order."""
        for src, dst in pairs:
            for cache in (self.k, self.v):
                cache[int(dst)] = (cache[int(src)] if int(src) in cache else self._fresh()).copy()

    def dense(self, which: str) -> np.ndarray:
        """The whole pool [num_blocks, N_kv, block_size, head_dim] as raw bits,
        unwritten blocks filled with the fill pattern."""
        cache = self.k if which == "k" else self.v
        out = np.full((self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim),
                      self.fill, dtype=STORAGE[self.kv_dtype])
        for b, arr in cache.items():
            out[b] = arr
        return out
