"""The C ABI on the host (no GPU): the library loads, exports what the header
declares, and its native allocator reproduces the oracle's tables, slots,
copy-on-write pairs, reference counts and free stack bit for bit."""
import json
import os
import random
import re

import numpy as np
import pytest
import torch

import workloads as W
from oracle import scenario as OS
from oracle.allocator import AllocError, BlockAllocator

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "sizing_examples.json")))


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    pkv.lib()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert "pkv_attention_decode" in names and "pkv_write" in names and "pkv_copy_blocks" in names
    handle = pkv.lib()
    for n in names:
        assert hasattr(handle, n), f"{n} declared in include/ but not exported"


def test_binding_covers_the_header():
    assert set(header_functions()) <= set(pkv.EXPORTED)


def test_block_bytes_and_budget():
    g = GOLD["block_bytes"]
    assert pkv.pkv_block_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["block_size"],
                               g["elem_bytes"]) == g["bytes"]
    assert pkv.pkv_block_bytes(0, 1, 1, 1, 1) == 0
    g = GOLD["pool_capacity"]
    n = pkv.pkv_num_blocks_for_budget(g["kv_budget_bytes"], g["block_bytes"])
    assert abs(n - g["approx_blocks"]) / g["approx_blocks"] < g["rel_tol"]
    assert pkv.pkv_dtype_bytes("e4m3") == 1 and pkv.pkv_dtype_bytes("bf16") == 2


def _compare(native: pkv.Pool, ref: BlockAllocator, live):
    assert native.num_free_blocks() == ref.num_free()
    assert native.free_stack().tolist() == ref.free_stack_top_first()
    for s in live:
        tab, ln = native.seq_table(s)
        assert tab.tolist() == ref.table(s) and ln == ref.context_len(s)
    for b in range(ref.num_blocks):
        assert native.block_refcount(b) == ref.block_refcount(b)
    # usage: live sequences, their tokens, blocks referenced (shared once)
    used = sum(1 for b in range(ref.num_blocks) if ref.block_refcount(b) > 0)
    assert native.usage() == (len(live), sum(ref.context_len(s) for s in live), used)


@pytest.mark.parametrize("seed", range(8))
def test_native_allocator_matches_oracle_on_random_ops(seed):
    rnd = random.Random(100 + seed)
    t = rnd.choice([16, 32])
    nb = rnd.choice([16, 64, 200])
    order = rnd.sample(range(nb), nb)
    native, ref = pkv.Pool(nb, t, order), BlockAllocator(nb, t, order)
    live, nxt = [], 0
    for step in range(400):
        op = rnd.random()
        if op < 0.15 or not live:
            native.seq_create(nxt)
            ref.create(nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.55:
            s, n = rnd.choice(live), rnd.randint(0, 2 * t + 3)
            try:
                exp = ref.append(s, n)
            except AllocError as e:
                with pytest.raises(pkv.PkvError) as got:
                    native.seq_append(s, n)
                assert got.value.code == e.code
            else:
                slots, cow = native.seq_append(s, n)
                assert slots.tolist() == exp[0] and [tuple(x) for x in cow.tolist()] == exp[1]
        elif op < 0.7:
            k = rnd.randint(1, 6)
            # half the batches may name a sequence more than once
            batch = rnd.choices(live, k=k) if rnd.random() < 0.5 else rnd.sample(live, min(len(live), k))
            try:
                exp = ref.append_batch(batch, 1)
            except AllocError as e:
                with pytest.raises(pkv.PkvError) as got:
                    native.batch_append(batch)
                assert got.value.code == e.code
            else:
                slots, cow = native.batch_append(batch)
                assert slots.tolist() == exp[0] and [tuple(x) for x in cow.tolist()] == exp[1]
        elif op < 0.82:
            parent = rnd.choice(live)
            native.seq_fork(parent, nxt)
            ref.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(rnd.randrange(len(live)))
            native.seq_free(s)
            ref.free_seq(s)
        if step % 25 == 0:
            _compare(native, ref, live)
    _compare(native, ref, live)


def test_batch_naming_a_sequence_twice_is_two_sequential_tokens():
    """The second token of a sequence named twice writes into the block its
    first token copied, so the batch needs one copy, not two: with one free
    block it is served exactly as the oracle's sequential appends serve it."""
    native, ref = pkv.Pool(4, 16), BlockAllocator(4, 16)
    for a in (native, ref):
        (a.seq_create if a is native else a.create)(1)
        (a.seq_append if a is native else a.append)(1, 20)
        (a.seq_fork if a is native else a.fork)(1, 2)
        (a.seq_create if a is native else a.create)(3)
        (a.seq_append if a is native else a.append)(3, 1)
    assert native.num_free_blocks() == ref.num_free() == 1
    want = ref.append_batch([2, 2], 1)
    slots, cow = native.batch_append([2, 2])
    assert slots.tolist() == want[0] == [52, 53] and [tuple(x) for x in cow.tolist()] == want[1]
    _compare(native, ref, [1, 2, 3])
    # a third token of sequence 2 would open a block: none is left, nothing changes
    native.seq_append(2, 10)
    ref.append(2, 10)
    with pytest.raises(pkv.PkvError) as e:
        native.batch_append([2, 2])
    with pytest.raises(AllocError) as f:
        ref.append_batch([2, 2], 1)
    assert e.value.code == f.value.code == "OUT_OF_BLOCKS"
    _compare(native, ref, [1, 2, 3])


@pytest.mark.parametrize("seed", range(12))
def test_batches_with_repeats_on_a_nearly_full_pool_match_oracle(seed):
    """Small pools, frequent mid-block forks and batches that repeat
    sequences: every batch append (served or refused) as the oracle's
    sequential appends, state compared after each."""
    rnd = random.Random(500 + seed)
    t, nb = 16, rnd.choice([6, 8, 12])
    native, ref = pkv.Pool(nb, t), BlockAllocator(nb, t)
    live, nxt = [], 0
    for step in range(300):
        op = rnd.random()
        if op < 0.2 or not live:
            ref.create(nxt)
            native.seq_create(nxt)
            live.append(nxt)
            n = rnd.randint(1, 2 * t)
            try:
                ref.append(nxt, n)
            except AllocError:
                with pytest.raises(pkv.PkvError):
                    native.seq_append(nxt, n)
            else:
                native.seq_append(nxt, n)
            nxt += 1
        elif op < 0.45:
            parent = rnd.choice(live)
            ref.fork(parent, nxt)
            native.seq_fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.55 and len(live) > 1:
            s = live.pop(rnd.randrange(len(live)))
            ref.free_seq(s)
            native.seq_free(s)
        else:
            batch = rnd.choices(live, k=rnd.randint(1, 5))
            try:
                exp = ref.append_batch(batch, 1)
            except AllocError as e:
                with pytest.raises(pkv.PkvError) as got:
                    native.batch_append(batch)
                assert got.value.code == e.code, (step, batch)
            else:
                slots, cow = native.batch_append(batch)
                assert slots.tolist() == exp[0], (step, batch)
                assert [tuple(x) for x in cow.tolist()] == exp[1], (step, batch)
        _compare(native, ref, live)


def test_errors_leave_state_unchanged():
    p = pkv.Pool(4, 16)
    p.seq_create(0)
    p.seq_append(0, 40)
    before = (p.free_stack().tolist(), p.seq_table(0)[0].tolist())
    with pytest.raises(pkv.PkvError) as e:
        p.seq_append(0, 40)
    assert e.value.code == "OUT_OF_BLOCKS"
    p.seq_create(1)
    p.seq_create(2)
    with pytest.raises(pkv.PkvError):
        p.batch_append([1, 2])
    assert (p.free_stack().tolist(), p.seq_table(0)[0].tolist()) == before
    assert p.seq_table(1)[1] == 0 and p.seq_table(2)[1] == 0
    with pytest.raises(pkv.PkvError) as e:
        p.seq_append(9, 1)
    assert e.value.code == "UNKNOWN_SEQ"
    with pytest.raises(pkv.PkvError) as e:
        p.seq_create(1)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(pkv.PkvError):
        pkv.Pool(3, 16, [0, 1, 1])
    with pytest.raises(pkv.PkvError):
        p.block_refcount(4)


def test_block_tables_padding_and_usage():
    p = pkv.Pool(8, 16, [7, 6, 5, 4, 3, 2, 1, 0])
    p.seq_create(5)
    p.seq_append(5, 20)
    p.seq_create(6)
    tables, ctx = p.block_tables([5, 6], 3)
    assert tables.tolist() == [[7, 6, -1], [-1, -1, -1]] and ctx.tolist() == [20, 0]
    with pytest.raises(pkv.PkvError):
        p.block_tables([5], 1)
    assert p.usage() == (2, 20, 2)


def test_block_tables_into_caller_buffers():
    p = pkv.Pool(8, 16, [7, 6, 5, 4, 3, 2, 1, 0])
    for s, n in ((5, 20), (6, 0), (9, 33)):
        p.seq_create(s)
        p.seq_append(s, n)
    want_t, want_c = p.block_tables([9, 5, 6], 4)
    for make in (lambda shape: np.full(shape, 77, np.int32),
                 lambda shape: torch.full(shape, 77, dtype=torch.int32)):
        t, c = make((3, 4)), make((3,))
        got = p.block_tables([9, 5, 6], 4, out=(t, c))
        assert got[0] is t and got[1] is c
        assert np.array_equal(np.asarray(t), want_t) and np.array_equal(np.asarray(c), want_c)
        # a failing call writes neither buffer
        t2, c2 = make((1, 1)), make((1,))
        with pytest.raises(pkv.PkvError):
            p.block_tables([9], 1, out=(t2, c2))
        assert np.asarray(t2).tolist() == [[77]] and np.asarray(c2).tolist() == [77]
    for bad in (np.zeros((3, 4), np.int64), np.zeros((4, 3), np.int32),
                np.zeros((4, 3), np.int32).T, torch.zeros((3, 4), dtype=torch.int64)):
        with pytest.raises(ValueError):
            p.block_tables([9, 5, 6], 4, out=(bad, np.zeros(3, np.int32)))


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_gqa_bf16", "prefix_fork_bf16", "long_mha_bf16",
                                  "fp8_churn"])
def test_workload_plans_match_oracle(name):
    w = W.get(name)
    native = PS.plan(w)
    ref = OS.build(w, write_seqs=[], scales={"k_inv_scale": 1.0, "v_inv_scale": 1.0})
    assert native.seq_ids == ref.seq_ids
    assert native.step_slots.tolist() == ref.step_slots
    assert [tuple(x) for x in native.cow_pairs.tolist()] == ref.cow_pairs
    for r, s in enumerate(ref.seq_ids):
        tab = ref.alloc.table(s)
        assert native.tables[r, :len(tab)].tolist() == tab
        assert np.all(native.tables[r, len(tab):] == -1)
        assert native.ctx_i32[r] == ref.ctx[r]
    assert native.pool.free_stack().tolist() == ref.alloc.free_stack_top_first()


def test_descriptor_head_scales_are_checked_before_any_launch():
    """Per-head scales belong to E4M3 caches: a 16-bit descriptor carrying a
    table is rejected by argument checking (no device work), an E4M3 one is
    accepted (an empty write), and the descriptor's layout matches the
    header's (six fields, the pointer last)."""
    import ctypes
    lib = pkv.lib()
    assert [f for f, _ in pkv.pkv_kv_desc._fields_][-1] == "head_scales"
    fake = ctypes.c_void_p(0x1000)            # never dereferenced: the calls stop at validation
    nothing = ctypes.c_void_p(0x2000)
    for dtype, want in (("bf16", pkv.PKV_ERR_INVALID_ARG), ("e4m3", pkv.PKV_OK)):
        d = pkv.kv_desc(16, 2, 128, 16, dtype)
        d.head_scales = fake.value
        st = lib.pkv_write(nothing, nothing, nothing, nothing, pkv.PKV_BF16, None, 0,
                           ctypes.byref(d), 1.0, 1.0, None)
        assert st == want, (dtype, st, lib.pkv_last_error())
    # the binding takes the table from a CUDA tensor only: a host address
    # would reach the kernels as a device pointer
    for bad in (torch.ones(4, 2), np.ones((4, 2), np.float32), torch.ones(2, 4, dtype=torch.float64)):
        with pytest.raises(ValueError):
            pkv.kv_desc(16, 2, 128, 16, "e4m3", head_scales=bad)
    d = pkv.kv_desc(16, 2, 128, 16, "e4m3")
    d.head_scales = 0x1002                    # not 4-byte aligned
    assert lib.pkv_write(nothing, nothing, nothing, nothing, pkv.PKV_BF16, None, 0,
                         ctypes.byref(d), 1.0, 1.0, None) == pkv.PKV_ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="the automatic partition follows the device's SM count; pinned for 152 SMs")
def test_automatic_partition_rule():
    """pkv_attention_partition(0) on the host's default of 152 SMs: one wave of
    split units when the pairs fit (Qwen-shaped batch: 1,536 tokens); when the
    (sequence, KV head) pairs fill two waves, half the longest context, at
    least 4,096 and at most 8,192 tokens."""
    bf16 = pkv.kv_desc(8500, 4, 128, 16, "bf16")
    e4m3 = pkv.kv_desc(65536, 8, 128, 16, "e4m3")
    fork = pkv.kv_desc(8192, 8, 128, 16, "bf16")
    assert pkv.pkv_attention_partition(64, 243, bf16) == 1536      # 452 units <= 456 slots
    assert pkv.pkv_attention_partition(512, 509, e4m3) == 4096     # longest 8,144 split in two
    assert pkv.pkv_attention_partition(256, 96, fork) == 4096      # 1,536-token contexts stay whole
    assert pkv.pkv_attention_partition(4096, 2048, e4m3) == 8192   # half of 32,768, capped
    assert pkv.pkv_attention_partition(64, 243, bf16, 512) == 512  # an explicit partition stands
    for n, mb in ((1, 1), (3, 700), (200, 40)):
        p = pkv.pkv_attention_partition(n, mb, bf16)
        assert p % 64 == 0 and 256 <= p <= 8192


@pytest.mark.parametrize("seed", range(6))
def test_incremental_block_tables_equal_full_ones(seed):
    """pkv_block_tables_update against pkv_block_tables after every step of a
    random stream of appends, batch appends, mid-block forks (copy-on-write),
    frees, ids created again, preemption, watermark admission and prefix-cache
    hits, with the batch reordered, shrunk and grown between steps and
    max_blocks changed once: tables and lengths equal bit for bit."""
    rnd = random.Random(seed)
    t = 16
    p = pkv.Pool(400, t)
    caching = seed % 2 == 1
    if caching:
        p.enable_prefix_cache()
    prompt = [rnd.randrange(50) for _ in range(8 * t)]
    live, next_id = [], 0
    rows = p.block_tables_rows(24, 40)
    for step in range(300):
        op = rnd.random()
        try:
            if op < 0.15 or not live:
                if caching and rnd.random() < 0.5:
                    n = rnd.randrange(1, len(prompt))
                    p.seq_create_cached(next_id, prompt[:n])
                    have = p.seq_table(next_id)[1]
                    p.seq_append_tokens(next_id, prompt[have:n])
                elif rnd.random() < 0.5:
                    p.seq_admit(next_id, rnd.randrange(0, 60), watermark_blocks=4)
                else:
                    p.seq_create(next_id)
                    p.seq_append(next_id, rnd.randrange(0, 60))
                live.append(next_id)
                next_id += 1
            elif op < 0.25:
                par = rnd.choice(live)
                p.seq_fork(par, next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.35:
                s = rnd.choice(live)
                p.seq_free(s)
                live.remove(s)
                if rnd.random() < 0.5:       # the same id again: a new sequence
                    p.seq_create(s)
                    p.seq_append(s, rnd.randrange(0, 40))
                    live.append(s)
            elif op < 0.45:
                _, _, gone = p.batch_append_preempt(list(live))
                live = [s for s in live if s not in gone]
            elif op < 0.7:
                p.seq_append(rnd.choice(live), rnd.randrange(1, 20))
            else:
                p.batch_append(rnd.sample(live, rnd.randrange(1, len(live) + 1)))
        except pkv.PkvError as e:
            assert e.code in ("OUT_OF_BLOCKS", "INVALID_ARG"), e
        while live and max(len(p.seq_table(s)[0]) for s in live) > rows.max_blocks:
            s = max(live, key=lambda x: len(p.seq_table(x)[0]))
            p.seq_free(s)
            live.remove(s)
        if step == 150:
            rows = p.block_tables_rows(24, 48)
        batch = rnd.sample(live, min(len(live), rnd.randrange(1, 25)))
        got_t, got_c = rows.update(batch)
        want_t, want_c = p.block_tables(batch, rows.max_blocks)
        assert np.array_equal(got_t.numpy(), want_t) and np.array_equal(got_c.numpy(), want_c), step


def test_incremental_block_tables_rewrite_only_what_can_change():
    """A row held for the same sequence is rewritten from its last entry on
    (a sentinel planted before it survives); a row that now holds another
    sequence, or whose state was reset, is rewritten whole; an error writes
    nothing."""
    p = pkv.Pool(64, 16)
    for s, n in ((1, 40), (2, 70)):
        p.seq_create(s)
        p.seq_append(s, n)
    rows = p.block_tables_rows(4, 8)
    rows.update([1, 2])
    rows.tables[0, 0] = 999                    # before row 0's last entry (index 2)
    p.seq_append(1, 30)                        # 70 tokens: entries 3 and 4 added
    t, c = rows.update([1, 2])
    assert t[0, 0] == 999 and t[0, 2:5].tolist() == p.seq_table(1)[0][2:5].tolist()
    assert c.tolist() == [70, 70]
    t, _ = rows.update([2, 1])                 # rows swapped: both rewritten whole
    want, _ = p.block_tables([2, 1], 8)
    assert np.array_equal(t.numpy(), want)
    rows.tables[1, 0] = 999
    rows.reset()
    t, _ = rows.update([2, 1])
    assert np.array_equal(t.numpy(), want)
    before = rows.tables.clone()
    with pytest.raises(pkv.PkvError):
        rows.update([2, 77])
    assert torch.equal(rows.tables, before)
    with pytest.raises(ValueError):
        rows.update([1, 2, 1, 2, 1])


C_CLIENT = r"""
#include "pkv.h"
#include <stdio.h>
int main(void) {
  pkv_pool* p = NULL;
  int64_t slots[40];
  int32_t cow[2], n_cow = 0, table[8], n_blocks = 0;
  int64_t ctx = 0;
  if (pkv_pool_create(8, 16, NULL, &p) != PKV_OK) return 1;
  if (pkv_seq_create(p, 1) != PKV_OK || pkv_seq_append(p, 1, 40, slots, cow, 1, &n_cow) != PKV_OK)
    return 2;
  if (pkv_seq_table(p, 1, table, 8, &n_blocks, &ctx) != PKV_OK) return 3;
  if (pkv_seq_append(p, 2, 1, slots, cow, 1, &n_cow) != PKV_ERR_UNKNOWN_SEQ) return 4;
  printf("%llu %d %lld %lld %d %d\n", (unsigned long long)pkv_block_bytes(28, 4, 128, 16, 2),
         n_blocks, (long long)ctx, (long long)slots[39], pkv_num_free_blocks(p),
         pkv_last_error()[0] != 0);
  pkv_pool_destroy(p);
  return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path):
    """The boundary is a C ABI: include/pkv.h compiles as strict C99 with no
    warning, and a C program links libpkv.so and drives the host allocator
    (no device call): the pages' 917,504-byte block, 3 blocks for 40 tokens,
    error codes and messages."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    pkv.lib()
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(pkv.LIB)
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src),
                        "-L", libdir, "-lpkv", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    # pool of 8 blocks, default order block 0 on top: 40 tokens -> blocks 0..2,
    # token 39 in block 2 at offset 7
    assert r.stdout.split() == ["917504", "3", "40", str(2 * 16 + 7), "5", "1"]


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("b,hq,n_kv,d,t,max_blocks,p", [
    (64, 28, 4, 128, 16, 243, 512), (64, 28, 4, 128, 16, 243, 1536), (3, 5, 1, 64, 32, 70, 64),
    (512, 64, 8, 128, 16, 509, 4096), (8, 32, 32, 128, 32, 1024, 512), (7, 12, 4, 64, 16, 9, 64)])
def test_workspace_bytes_follow_the_documented_layout(b, hq, n_kv, d, t, max_blocks, p):
    """Split-K workspace for an explicit partition P: int32 arrival counters
    [B][N_kv], then fp32 maxima and sums [B][Hq][S] and unnormalised outputs
    [B][Hq][S][D], each part 256-byte aligned, S = ceil(max_blocks * T / P);
    nothing when one split covers every sequence."""
    desc = pkv.kv_desc(1000, n_kv, d, t, "bf16")
    s = -(-max_blocks * t // p)
    n = b * hq * s
    want = 0 if s <= 1 else (_align256(4 * b * n_kv) + 2 * _align256(4 * n) + _align256(4 * n * d))
    assert pkv.pkv_attention_workspace_bytes(b, hq, max_blocks, desc, p) == want


def test_workspace_bytes_reject_bad_sizes():
    desc = pkv.kv_desc(1000, 4, 128, 16, "bf16")
    for args in ((64, 28, 243, 100), (64, 28, 243, 48), (64, 28, 243, -512), (0, 28, 243, 512),
                 (64, 0, 243, 512), (64, 28, 0, 512)):
        assert pkv.pkv_attention_workspace_bytes(*args[:3], desc, args[3]) == 0, args
    desc32 = pkv.kv_desc(1000, 4, 128, 32, "bf16")
    assert pkv.pkv_attention_workspace_bytes(4, 28, 100, desc32, 64) > 0   # 64 is a multiple of 32


def test_automatic_workspace_is_the_resolved_partitions():
    desc = pkv.kv_desc(8500, 4, 128, 16, "bf16")
    p = pkv.pkv_attention_partition(64, 243, desc)
    assert p == 1536
    assert pkv.pkv_attention_workspace_bytes(64, 28, 243, desc, 0) == \
        pkv.pkv_attention_workspace_bytes(64, 28, 243, desc, p)
