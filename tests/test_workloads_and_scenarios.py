"""The seeded workloads and the oracle's scenario builder: structure of each
synthetic configuration (no GPU)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import scenario as S
from oracle import sizing


def test_generators_are_deterministic_and_position_keyed():
    w = W.get("qwen_gqa_bf16")
    k, v = W.kv_for_seq(w, 3, 40)
    k2, v2 = W.kv_for_seq(w, 3, 15, first_pos=25)
    assert torch.equal(k[25:], k2) and torch.equal(v[25:], v2)
    assert torch.equal(W.q_for_seq(w, 5), W.q_for_seq(w, 5))
    assert not torch.equal(W.q_for_seq(w, 5), W.q_for_seq(w, 6))
    assert k.dtype == torch.bfloat16 and k.shape == (40, 4, 128)


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_gqa_bf16", "long_mha_bf16", "fp8_churn"])
def test_context_lengths_in_range_and_fit_pool(name):
    w = W.get(name)
    ctx = W.context_lens(w)
    lo, hi = w.ctx_range
    assert len(ctx) == w.num_seqs and ctx.min() >= lo and ctx.max() <= hi
    assert sum(sizing.blocks_for_tokens(int(c), w.block_size) for c in ctx) <= w.num_blocks


def test_spiked_keys():
    w = W.get("long_mha_bf16")
    k, _ = W.kv_for_seq(w, 0, 200)
    norms = k.float().norm(dim=-1).mean(dim=-1)
    spiked = [p for p in range(200) if (p + 1) % 97 == 0]
    assert spiked == [96, 193]
    assert all(norms[p] > 4 * norms.median() for p in spiked)


def test_fork_layout():
    w = W.get("prefix_fork_bf16")
    lay = W.fork_layout(w)
    assert lay["num_children"] == 64 and lay["num_parents"] == 192
    prior = w.prefix_len + lay["tails"] - 1
    assert np.all(prior[lay["parent_of_child"]] % w.block_size != 0)
    assert len(set(lay["parent_of_child"].tolist())) == 64


def test_fp8_scales_cover_amax():
    sc = W.fp8_scales(6.0, 5.5)
    assert np.float32(6.0) * np.float32(sc["k_inv_scale"]) <= np.float32(448.0) * (1 + 1e-6)
    assert abs(sc["k_scale"] * 448 - 6.0) < 1e-5


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_gqa_bf16"])
def test_scenario_tables_cover_context(name):
    w = W.get(name)
    scn = S.build(w, write_seqs=[0, 1])
    for r, s in enumerate(scn.seq_ids):
        tab = scn.alloc.table(s)
        assert scn.alloc.context_len(s) == scn.ctx[r]
        assert len(tab) == sizing.blocks_for_tokens(int(scn.ctx[r]), w.block_size)
        p = int(scn.ctx[r]) - 1
        assert scn.step_slots[r] == tab[p // w.block_size] * w.block_size + p % w.block_size
    assert scn.cow_pairs == []


def test_prefix_fork_scenario_structure():
    w = W.get("prefix_fork_bf16")
    scn = S.build(w, write_seqs=[0, 64])
    a = scn.alloc
    prefix_blocks = a.table(0)[:64]
    for b in prefix_blocks:
        assert a.block_refcount(b) == 256
    assert len(scn.cow_pairs) == 64
    for c in range(64):
        child = scn.seq_ids[c]
        assert a.table(child)[:64] == prefix_blocks
    # after the step every last block is owned by one sequence
    for s in scn.seq_ids:
        assert a.block_refcount(a.table(s)[-1]) == 1


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_gqa_bf16", "long_mha_bf16", "fp8_churn",
                                  "prefix_fork_bf16"])
def test_unique_kv_bytes(name):
    """The roofline's algorithmic bytes: with no shared block they are the
    logical bytes; for the prefix fork, the distinct cached tokens are the
    prefix once, every parent's tail, and per child the slots of its own
    copied last block (positions floor(prior / T) * T .. prior)."""
    from paged_kv_cache_137_gb300 import scenario as PS
    w = W.get(name)

    class Host:  # the byte counts need the plan only, not the device buffers
        plan = PS.plan(w)

    unique = PS.DeviceScenario.kv_unique_bytes(Host)
    logical = PS.DeviceScenario.kv_bytes(Host)
    per_token = 2 * w.num_kv_heads * w.head_dim * w.kv_bytes
    if w.ctx_dist != "prefix_fork":
        assert unique == logical == per_token * int(W.context_lens(w).sum())
        return
    f = W.fork_layout(w)
    prior = w.prefix_len + f["tails"] - 1
    tokens = w.prefix_len + int(f["tails"].sum()) + int((prior[f["parent_of_child"]] % w.block_size + 1).sum())
    assert unique == per_token * tokens
    assert logical == per_token * int(f["ctx"].sum()) > 6 * unique


def test_churn_scrambles_but_returns_every_block():
    w = W.get("fp8_churn")
    from oracle.allocator import BlockAllocator
    a = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    top_before = a.free_stack_top_first()[:100]
    S.apply_churn(a, *W.churn_ops(w), w.block_size)
    assert a.num_free() == w.num_blocks
    assert a.free_stack_top_first()[:100] != top_before
