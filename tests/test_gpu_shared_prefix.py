"""GPU parity of the shared-prefix decode path against the CPU oracle.

A batch whose sequences all map the same leading blocks (forks of one
prompt: "PagedAttention Memory Management", "Complex Topologies and Memory
Sharing"; the katajob Q&A, "Sharing, the second dividend") is decoded by
pkv_decode_step_shared_prefix: a tcgen05 pass attends every sequence's
queries to the shared blocks once, the tail queue (or, where it does not
apply, the split kernel's narrow forms) attends the rest of each context, and
a merge kernel combines the partials.  The result is plain attention, so it is
compared with
the oracle at the decode tolerances; the reduction is split differently from
the plain path, so the two paths agree within rounding, not bit for bit (the
foundry page, "Effect": reusing shared blocks changes how the attention
reduction is tiled).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import scenario as OS

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

from test_gpu_parity import check_close, oracle_out, pool_bits, oracle_pool_bits

pytestmark = pytest.mark.gpu

BASE = W.get("prefix_fork_bf16")
CASES = {
    # 48 sequences x 4 heads = 192 rows: one full 128-row tile and a partial
    # second; a 288-token prompt (18 blocks, 4.5 key tiles)
    "pfx_rows192": W.scaled(BASE, num_seqs=48, num_blocks=2048, prefix_len=288, tail_range=(1, 200)),
    # 80 sequences: 320 rows, two row pairs; a 1,024-token prefix
    "pfx_rows320": W.scaled(BASE, num_seqs=80, num_blocks=2048, prefix_len=1024, tail_range=(1, 100),
                            seed=77),
    # 16 sequences: 64 rows, one partial tile; 96 shared tokens
    "pfx_rows64": W.scaled(BASE, num_seqs=16, num_blocks=256, prefix_len=96, tail_range=(1, 60)),
    "pfx_f16": W.scaled(BASE, num_seqs=40, num_blocks=2048, prefix_len=528, tail_range=(1, 90),
                        kv_dtype="f16", q_dtype="f16", seed=78),
    "pfx_t32": W.scaled(BASE, num_seqs=40, num_blocks=1024, prefix_len=704, tail_range=(1, 150),
                        block_size=32, seed=79),
    "pfx_e4m3": W.scaled(BASE, num_seqs=40, num_blocks=2048, prefix_len=592, tail_range=(1, 120),
                         kv_dtype="e4m3", q_dtype="bf16", seed=80),
    # group 8 (64 query / 8 KV heads): 8 rows per sequence
    "pfx_g8": W.scaled(BASE, num_seqs=24, num_q_heads=64, num_kv_heads=8, num_blocks=2048,
                       prefix_len=400, tail_range=(1, 80), seed=81),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


@pytest.fixture(autouse=True)
def clean_status():
    pkv.pkv_device_status(clear=True)
    yield


def scales_of(w):
    """E4M3 scales: the prefix-fork inputs are N(0,1), so a fixed amax of 6
    (both sides quantise with the same scale, saturating beyond it)."""
    return W.fp8_scales(6.0, 6.0) if w.kv_dtype == "e4m3" else {}


def shared(w, partition=None):
    sc = scales_of(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc, partition_tokens=partition, shared_prefix=True)
    assert dev.prefix_blocks == dev.plan.shared_prefix_blocks > 0
    return dev, sc


@pytest.mark.parametrize("name", list(CASES))
def test_shared_prefix_step_matches_oracle(name):
    w = CASES[name]
    dev, sc = shared(w)
    out = dev.step()
    torch.cuda.synchronize()
    ref = OS.build(w, scales=sc)
    # copy-on-write copies and the fused slot write: every pool byte exact
    assert np.array_equal(pool_bits(dev.k_cache).reshape(-1), oracle_pool_bits(ref, "k"))
    assert np.array_equal(pool_bits(dev.v_cache).reshape(-1), oracle_pool_bits(ref, "v"))
    check_close(out.double().cpu().numpy(), oracle_out(ref), w.kv_dtype)
    assert pkv.pkv_device_status() == 0


@pytest.mark.parametrize("partition", [0, 64, 128, 512, 1024])
def test_shared_prefix_with_split_tails(partition):
    """Tails split over several units (the tail queue up to 32 tiles a unit,
    the split kernel past it: 64 and 1,024 tokens): the merge kernel combines
    the tail splits with the prefix pass's partials."""
    w = CASES["pfx_rows192"]
    dev, sc = shared(w, partition)
    out = dev.step()
    torch.cuda.synchronize()
    check_close(out.double().cpu().numpy(), oracle_out(OS.build(w, scales=sc)), w.kv_dtype)
    n = len(dev.plan.seq_ids) * w.num_kv_heads
    assert torch.count_nonzero(dev.workspace[: 4 * n + 8]).item() == 0   # counters back at zero


def test_shared_and_plain_paths_agree():
    """The same device state through the shared-prefix path and the plain
    path: both within tolerance of the oracle, and of each other."""
    w = CASES["pfx_rows320"]
    dev, sc = shared(w)
    dev.copy_blocks()
    dev.write_step()
    a = dev.attend().double().cpu().numpy().copy()
    ws = pkv.workspace_for(len(dev.plan.seq_ids), w.num_q_heads, dev.plan.max_blocks, dev.desc, 0)
    out = torch.empty_like(dev.q)
    pkv.pkv_attention_decode(out, dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.ctx, dev.desc,
                             dev.softmax_scale, partition_tokens=0, workspace=ws)
    b = out.double().cpu().numpy()
    ref = oracle_out(OS.build(w, scales=sc))
    check_close(a, ref, "bf16")
    check_close(b, ref, "bf16")
    assert np.abs(a - b).max() <= 2e-2


def test_shared_prefix_physical_permutation_is_bit_identical():
    """Relocating every block (the pool permuted, the tables renamed) leaves
    the shared-prefix path's output unchanged bit for bit: the split
    boundaries depend only on logical positions."""
    w = CASES["pfx_rows192"]
    dev, sc = shared(w)
    dev.copy_blocks()
    dev.write_step()
    a = dev.attend().clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5)).cuda()
    k2 = torch.empty_like(dev.k_cache)
    v2 = torch.empty_like(dev.v_cache)
    k2[perm] = dev.k_cache
    v2[perm] = dev.v_cache
    t = dev.tables.long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], t).int()
    out = torch.empty_like(dev.q)
    pkv.pkv_attention_decode_shared_prefix(out, dev.q, k2, v2, t2, dev.ctx, dev.desc, dev.prefix_blocks,
                                           dev.softmax_scale, partition_tokens=dev.partition,
                                           workspace=dev.workspace)
    torch.cuda.synchronize()
    assert not torch.equal(t2, dev.tables)
    assert torch.equal(a.view(torch.int16), out.view(torch.int16))


def test_broken_prefix_declaration_gives_nan_and_status():
    """A row that does not map the declared shared blocks, and a row whose
    context ends inside the prefix, get NaN and set their device error bits;
    the other rows stay correct."""
    w = CASES["pfx_rows192"]
    dev, sc = shared(w)
    dev.copy_blocks()
    dev.write_step()
    ref = oracle_out(OS.build(w, scales=sc))
    tables = dev.tables.clone()
    ctx = dev.ctx.clone()
    tables[3, 1] = int(dev.plan.tables[3, 2])          # a valid block, not the shared one
    ctx[5] = dev.prefix_blocks * w.block_size           # context ends at the prefix
    out = torch.empty_like(dev.q)
    pkv.pkv_attention_decode_shared_prefix(out, dev.q, dev.k_cache, dev.v_cache, tables, ctx, dev.desc,
                                           dev.prefix_blocks, dev.softmax_scale, workspace=dev.workspace)
    torch.cuda.synchronize()
    flags = pkv.pkv_device_status(clear=True)
    assert flags == pkv.PKV_DEVICE_BAD_SHARED_PREFIX | pkv.PKV_DEVICE_BAD_LENGTH
    got = out.double().cpu().numpy()
    assert np.isnan(got[3]).all() and np.isnan(got[5]).all()
    rows = [r for r in range(len(got)) if r not in (3, 5)]
    check_close(got, ref, "bf16", rows=rows)


def test_shared_prefix_full_size():
    """The prefix-fork workload at full size (256 sequences, 1,024 shared
    tokens) in the launch configuration the benchmark times, every row
    against the oracle."""
    w = W.get("prefix_fork_bf16")
    dev = PS.materialize(PS.plan(w), "cuda")
    assert dev.prefix_blocks == 64
    out = dev.step()
    torch.cuda.synchronize()
    ref = OS.build(w)
    check_close(out.double().cpu().numpy(), oracle_out(ref), "bf16")
    assert pkv.pkv_device_status() == 0


@pytest.mark.parametrize("name,kernel", [("pfx_rows192", "auto"), ("pfx_rows192", "tc"),
                                         ("pfx_t32", "auto")])
def test_tail_wait_give_up_gives_nan_and_status_then_recovers(name, kernel):
    """The tail kernels' failure path behind a shared prefix (the tail queue
    at block size 16, the one-warp split form when the split kernel is
    forced, the two-warp form at 32), run on purpose: with a stage-wait limit
    of 0 every tail CTA gives up at its first stage wait, drains its copies in
    flight (its own bounded limit), writes NaN partials (the queue form for
    every unit it holds or claims afterwards) and sets
    PKV_DEVICE_WAIT_TIMEOUT; the merge kernel carries the NaN to every output
    whose context extends past the prefix, and the counters end at zero.  The
    next call, with the normal limit, is correct."""
    w = CASES[name]
    dev, sc = shared(w)
    dev.copy_blocks()
    try:
        pkv.pkv_set_attention_kernel(kernel)
        pkv.pkv_set_stage_wait_limit(0)
        out = dev.decode_step().clone()
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_stage_wait_limit(50_000_000)
        pkv.pkv_set_attention_kernel("auto")
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVICE_WAIT_TIMEOUT
    assert torch.isnan(out).all()   # every context extends past the prefix
    n = len(dev.plan.seq_ids) * w.num_kv_heads
    # counters, the exit count and the queue's claim counter
    assert torch.count_nonzero(dev.workspace[: 4 * n + 8]).item() == 0
    out = dev.decode_step()
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    ref = OS.build(w, scales=sc)
    check_close(out.double().cpu().numpy(), oracle_out(ref), w.kv_dtype)


@pytest.mark.parametrize("name,partition", [("pfx_rows192", 0), ("pfx_rows192", 128),
                                            ("pfx_rows320", 512), ("pfx_f16", 0), ("pfx_g8", 256)])
def test_tail_queue_equals_split_kernel_bit_for_bit(name, partition):
    """The tail queue (one-warp CTAs taking units longest first) and the
    one-warp split kernel (one CTA per unit) attend the same splits in the
    same tile order with the same arithmetic: the outputs are the same bits,
    and so are the step's pool writes."""
    w = CASES[name]
    outs, pools = [], []
    for kernel in ("auto", "tc"):
        dev, sc = shared(w, partition)
        try:
            pkv.pkv_set_attention_kernel(kernel)
            out = dev.step()
            torch.cuda.synchronize()
        finally:
            pkv.pkv_set_attention_kernel("auto")
        outs.append(out.clone())
        pools.append((dev.k_cache.clone(), dev.v_cache.clone()))
        assert pkv.pkv_device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(pools[0][0].view(torch.uint8), pools[1][0].view(torch.uint8))
    assert torch.equal(pools[0][1].view(torch.uint8), pools[1][1].view(torch.uint8))
    check_close(outs[0].double().cpu().numpy(), oracle_out(OS.build(w, scales=sc)), w.kv_dtype)
