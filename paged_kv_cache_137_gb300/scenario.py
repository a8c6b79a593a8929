"""The synthetic decode workloads driven through libpkv.

``plan`` runs a workload's allocation on the native allocator (host only):
optional alloc/free churn, a prefill of every sequence's prior tokens, forks,
and the decode step's one-token append with its copy-on-write pairs.
``materialize`` then builds the device state: the K/V pool filled through the
slot-write kernel, q, block tables, context lengths and the step's new K/V.
``DeviceScenario.step`` is one decode step of the hot path: block copies, slot
write, decode attention.

Workload rules (the pages describe the mechanism, not these workloads):
prefill appends a sequence's ctx - 1 prior tokens in one call, sequences in
batch order; the step appends one token per sequence in batch order.  Churn
operation i allocates a fresh one-block sequence when coin[i] < 0.5 and a block
is free (or nothing is live), else finishes the live churn sequence at index
floor(pick[i] * live) of the live list (allocation order); afterwards every
churn sequence is finished in list order.  Prefix fork: parent 0 prefills the
prefix, parents 1.. fork it, each parent prefills its tail, each child forks
its parent; the batch is children then parents.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

import workloads as W

from . import (Pool, empty_cache, kv_desc, pkv_attention_decode, pkv_attention_decode_shared_prefix,
               pkv_copy_blocks, pkv_decode_step, pkv_decode_step_shared_prefix, pkv_write,
               prepare_copy_blocks, prepare_decode_step, shared_prefix_workspace_for,
               workspace_for)

CHURN_ID0 = 1 << 40
POISON_BYTE = 0xFF


@dataclass
class PrefillWrite:
    seq: int            # stream index of the K/V draws
    first_pos: int
    n_tokens: int
    slots: np.ndarray
    prefix: bool = False


@dataclass
class Plan:
    w: W.Workload
    pool: Pool
    seq_ids: list
    ctx: np.ndarray
    prefill: list
    step_slots: np.ndarray
    cow_pairs: np.ndarray
    max_blocks: int
    tables: np.ndarray = field(default=None)
    ctx_i32: np.ndarray = field(default=None)
    shared_prefix_blocks: int = 0   # leading blocks every sequence of the batch maps


def churn(pool: Pool, coin, pick, block_size: int):
    live, nxt = [], CHURN_ID0
    for c, p in zip(coin, pick):
        if (c < 0.5 and pool.num_free_blocks() > 0) or not live:
            pool.seq_create(nxt)
            pool.seq_append(nxt, block_size)
            live.append(nxt)
            nxt += 1
        else:
            pool.seq_free(live.pop(int(p * len(live))))
    for s in live:
        pool.seq_free(s)


def plan(w: W.Workload) -> Plan:
    pool = Pool(w.num_blocks, w.block_size, W.free_order(w))
    if w.churn:
        churn(pool, *W.churn_ops(w), w.block_size)
    ctx = np.asarray(W.context_lens(w), dtype=np.int64)
    writes = []
    if w.ctx_dist == "prefix_fork":
        lay = W.fork_layout(w)
        n_par, n_ch = lay["num_parents"], lay["num_children"]
        seq_ids = [n_par + c for c in range(n_ch)] + list(range(n_par))
        pool.seq_create(0)
        slots, _ = pool.seq_append(0, w.prefix_len)
        writes.append(PrefillWrite(-1, 0, w.prefix_len, slots, prefix=True))
        for p in range(1, n_par):
            pool.seq_fork(0, p)
        for p in range(n_par):
            n = int(lay["tails"][p]) - 1
            slots, _ = pool.seq_append(p, n)
            writes.append(PrefillWrite(p, w.prefix_len, n, slots))
        for c in range(n_ch):
            pool.seq_fork(int(lay["parent_of_child"][c]), n_par + c)
    else:
        seq_ids = list(range(w.num_seqs))
        for r, s in enumerate(seq_ids):
            pool.seq_create(s)
            slots, _ = pool.seq_append(s, int(ctx[r]) - 1)
            writes.append(PrefillWrite(s, 0, int(ctx[r]) - 1, slots))
    step_slots, cow = pool.batch_append(seq_ids)
    max_blocks = max(1, max(-(-int(c) // w.block_size) for c in ctx))
    tables, ctx32 = pool.block_tables(seq_ids, max_blocks)
    return Plan(w=w, pool=pool, seq_ids=seq_ids, ctx=ctx, prefill=writes, step_slots=step_slots,
                cow_pairs=cow, max_blocks=max_blocks, tables=tables, ctx_i32=ctx32,
                shared_prefix_blocks=pool.shared_prefix_blocks(seq_ids))


@dataclass
class DeviceScenario:
    plan: Plan
    desc: object
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor
    out: torch.Tensor
    tables: torch.Tensor
    ctx: torch.Tensor
    step_slots: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    workspace: torch.Tensor | None
    scales: dict             # per-tensor E4M3 scale arguments ({} with per-head scales in desc)
    partition: int           # partition_tokens passed to the decode call (0 = automatic)
    softmax_scale: float
    prefix_blocks: int = 0   # > 0: the decode calls attend this shared prefix once for all rows

    def copy_blocks(self, stream=None):
        pkv_copy_blocks([self.k_cache], [self.v_cache], self.plan.cow_pairs, self.desc, stream)

    def write_step(self, stream=None):
        pkv_write(self.k_cache, self.v_cache, self.k_new, self.v_new, self.step_slots, self.desc,
                  self.scales.get("k_inv_scale", 1.0), self.scales.get("v_inv_scale", 1.0), stream)

    def attend(self, stream=None, partition_tokens=None, out=None, workspace=None):
        p = self.partition if partition_tokens is None else partition_tokens
        ws = self.workspace if workspace is None else workspace
        if self.prefix_blocks:
            return pkv_attention_decode_shared_prefix(
                self.out if out is None else out, self.q, self.k_cache, self.v_cache, self.tables,
                self.ctx, self.desc, self.prefix_blocks, self.softmax_scale,
                self.scales.get("k_scale", 1.0), self.scales.get("v_scale", 1.0), p, ws, stream)
        return pkv_attention_decode(self.out if out is None else out, self.q, self.k_cache,
                                    self.v_cache, self.tables, self.ctx, self.desc,
                                    self.softmax_scale, self.scales.get("k_scale", 1.0),
                                    self.scales.get("v_scale", 1.0), p, ws, stream)

    def decode_step(self, stream=None, out=None):
        """Slot write of the step's token fused with attention (pkv_decode_step,
        or pkv_decode_step_shared_prefix over a shared prefix)."""
        if self.prefix_blocks:
            return pkv_decode_step_shared_prefix(
                self.out if out is None else out, self.q, self.k_cache, self.v_cache, self.k_new,
                self.v_new, self.tables, self.ctx, self.desc, self.prefix_blocks, self.softmax_scale,
                self.scales.get("k_scale", 1.0), self.scales.get("v_scale", 1.0),
                self.scales.get("k_inv_scale", 1.0), self.scales.get("v_inv_scale", 1.0),
                self.partition, self.workspace, stream)
        return pkv_decode_step(self.out if out is None else out, self.q, self.k_cache, self.v_cache,
                               self.k_new, self.v_new, self.tables, self.ctx, self.desc,
                               self.softmax_scale, self.scales.get("k_scale", 1.0),
                               self.scales.get("v_scale", 1.0), self.scales.get("k_inv_scale", 1.0),
                               self.scales.get("v_inv_scale", 1.0), self.partition, self.workspace,
                               stream)

    def step(self, stream=None):
        """One decode step of the hot path: block copies, then the slot write
        fused with attention."""
        self.copy_blocks(stream)
        return self.decode_step(stream)

    def prepare_step(self):
        """step() as Prepared calls on this scenario's buffers: a function of
        the stream (a raw cudaStream_t int or a torch stream) that launches the
        block copies, then the fused slot write and attention."""
        copies = prepare_copy_blocks([self.k_cache], [self.v_cache], self.plan.cow_pairs, self.desc)
        decode = prepare_decode_step(
            self.out, self.q, self.k_cache, self.v_cache, self.k_new, self.v_new, self.tables,
            self.ctx, self.desc, self.softmax_scale, self.scales.get("k_scale", 1.0),
            self.scales.get("v_scale", 1.0), self.scales.get("k_inv_scale", 1.0),
            self.scales.get("v_inv_scale", 1.0), self.partition, self.workspace,
            prefix_blocks=self.prefix_blocks or None)

        def run(stream):
            if copies is not None:
                copies(stream)
            decode(stream)
        return run

    def kv_bytes(self) -> int:
        """Logical K/V bytes one attention call serves: every sequence's
        context once (a block shared by n sequences counts n times)."""
        w = self.plan.w
        return int(2 * int(self.plan.ctx.sum()) * w.num_kv_heads * w.head_dim * w.kv_bytes)

    def kv_unique_bytes(self) -> int:
        """K/V bytes of the distinct cache slots the call reads: each stored
        element once, however many sequences share its block (equal to
        kv_bytes() when no block is shared)."""
        w, tab, ctx = self.plan.w, self.plan.tables, self.plan.ctx
        t = w.block_size
        filled = {}  # physical block -> slots read in it (the longest use)
        for r, c in enumerate(ctx):
            c = int(c)
            for j in range(-(-c // t)):
                b = int(tab[r, j])
                filled[b] = max(filled.get(b, 0), min(t, c - j * t))
        return int(2 * sum(filled.values()) * w.num_kv_heads * w.head_dim * w.kv_bytes)


def _kv_of(w, pw: PrefillWrite):
    if pw.prefix:
        return W.prefix_kv(w)
    return W.kv_for_seq(w, pw.seq, pw.n_tokens, first_pos=pw.first_pos)


def use_shared_prefix(p: Plan) -> bool:
    """Whether the decode calls take the shared-prefix path by default: a
    prefix of at least 256 tokens shared by enough (sequence, head) rows to
    fill one 128-row tensor-core tile per KV head."""
    w = p.w
    return (p.shared_prefix_blocks * w.block_size >= 256 and len(p.seq_ids) * w.group >= 128
            and w.head_dim == 128 and w.kv_dtype != "f32")


def materialize(p: Plan, device="cuda", scales: dict | None = None, chunk_tokens: int = 1 << 19,
                partition_tokens: int | None = None, shared_prefix: bool | None = None) -> DeviceScenario:
    """The device state of a plan.  shared_prefix: take the shared-prefix
    decode path over the plan's shared blocks (None: use_shared_prefix)."""
    w = p.w
    scales = dict(scales or {})
    if w.kv_dtype == "e4m3" and "k_inv_scale" not in scales:
        raise ValueError("an E4M3 cache needs its scales")
    head_scales = None
    if np.ndim(scales.get("k_scale", 1.0)) > 0:
        # per-KV-head scales go in the descriptor; the per-tensor arguments
        # of every call are then ignored (left at 1)
        rows = [np.asarray(scales[n], dtype=np.float32)
                for n in ("k_scale", "v_scale", "k_inv_scale", "v_inv_scale")]
        head_scales = torch.from_numpy(np.stack(rows)).to(device)
        scales = {}
    desc = kv_desc(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.kv_dtype, head_scales)
    k_cache, v_cache = empty_cache(desc, device, fill_byte=POISON_BYTE)
    kinv, vinv = scales.get("k_inv_scale", 1.0), scales.get("v_inv_scale", 1.0)

    pend_k, pend_v, pend_s, n_pend = [], [], [], 0

    def flush():
        nonlocal pend_k, pend_v, pend_s, n_pend
        if not n_pend:
            return
        k = torch.cat(pend_k).to(device)
        v = torch.cat(pend_v).to(device)
        s = torch.from_numpy(np.concatenate(pend_s)).to(device)
        pkv_write(k_cache, v_cache, k, v, s, desc, kinv, vinv)
        pend_k, pend_v, pend_s, n_pend = [], [], [], 0

    for pw in p.prefill:
        if pw.n_tokens == 0:
            continue
        k, v = _kv_of(w, pw)
        pend_k.append(k)
        pend_v.append(v)
        pend_s.append(np.asarray(pw.slots, dtype=np.int64))
        n_pend += pw.n_tokens
        if n_pend >= chunk_tokens:
            flush()
    flush()

    news = [W.kv_for_seq(w, s, 1, first_pos=int(p.ctx[r]) - 1) for r, s in enumerate(p.seq_ids)]
    k_new = torch.cat([k for k, _ in news]).to(device)
    v_new = torch.cat([v for _, v in news]).to(device)
    q = torch.stack([W.q_for_seq(w, s) for s in p.seq_ids]).to(device)
    part = w.partition_tokens if partition_tokens is None else partition_tokens
    if shared_prefix is None:
        shared_prefix = use_shared_prefix(p)
    pfx = p.shared_prefix_blocks if shared_prefix else 0
    if pfx:
        ws = shared_prefix_workspace_for(len(p.seq_ids), w.num_q_heads, p.max_blocks, desc, pfx, part,
                                         device)
    else:
        ws = workspace_for(len(p.seq_ids), w.num_q_heads, p.max_blocks, desc, part, device)
    return DeviceScenario(
        plan=p, desc=desc, k_cache=k_cache, v_cache=v_cache, q=q, out=torch.empty_like(q),
        tables=torch.from_numpy(p.tables).to(device), ctx=torch.from_numpy(p.ctx_i32).to(device),
        step_slots=torch.from_numpy(np.asarray(p.step_slots, dtype=np.int64)).to(device),
        k_new=k_new, v_new=v_new, workspace=ws, scales=scales,
        partition=part,
        softmax_scale=1.0 / math.sqrt(w.head_dim), prefix_blocks=pfx)
