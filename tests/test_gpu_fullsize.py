"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times: the GPU runs the whole batch; the oracle
recomputes every sequence of the Qwen-shaped batch and a sample of the
others' one by one (their pool blocks bit-exact, their outputs within
tolerance)."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import scenario as OS

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

from test_gpu_parity import TOL, scales_for

pytestmark = pytest.mark.gpu

FULL = ["tiny_fp32", "qwen_gqa_bf16", "prefix_fork_bf16", "long_mha_bf16", "fp8_churn"]


def sample_rows(ctx, k=4, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, len(ctx) - 1, int(np.argmax(ctx)), int(np.argmin(ctx))}
    rows |= set(rng.choice(len(ctx), size=min(k, len(ctx)), replace=False).tolist())
    return sorted(rows)


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    w = W.get(name)
    sc = scales_for(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc)
    dev.copy_blocks()
    dev.write_step()
    outs = {}
    try:
        for k in ("simt", "tc") if w.kv_dtype != "f32" else ("simt",):
            pkv.pkv_set_attention_kernel(k)   # the workspace size follows the kernel choice
            if dev.prefix_blocks:
                ws = pkv.shared_prefix_workspace_for(len(dev.plan.seq_ids), w.num_q_heads,
                                                     dev.plan.max_blocks, dev.desc, dev.prefix_blocks,
                                                     dev.partition)
            else:
                ws = pkv.workspace_for(len(dev.plan.seq_ids), w.num_q_heads, dev.plan.max_blocks,
                                       dev.desc, dev.partition)
            outs[k] = dev.attend(workspace=ws).double().cpu().numpy().copy()
    finally:
        pkv.pkv_set_attention_kernel("auto")
    torch.cuda.synchronize()
    # the headline workload whole, the others on sampled rows
    rows = list(range(len(dev.plan.ctx))) if name == "qwen_gqa_bf16" else sample_rows(dev.plan.ctx)
    ref_scn = OS.build(w, write_seqs=rows, scales=sc)
    ref = OA.paged_attention_decode(ref_scn.q_f64(), ref_scn.pool, ref_scn.tables, ref_scn.ctx,
                                    1.0 / math.sqrt(w.head_dim), sc.get("k_scale", 1.0),
                                    sc.get("v_scale", 1.0), seqs=rows)
    max_tol, mean_tol = TOL[w.kv_dtype]
    for k, got in outs.items():
        assert not np.isnan(got).any(), k
        err = np.abs(got[rows] - ref[rows])
        assert err.max() <= max_tol, f"{k}: max abs error {err.max():.3g}"
        if mean_tol is not None:
            assert err.mean() <= mean_tol, f"{k}: mean abs error {err.mean():.3g}"
    # the sampled sequences' blocks hold exactly the oracle's bytes
    kc = dev.k_cache.view(torch.uint8)
    vc = dev.v_cache.view(torch.uint8)
    for r in rows:
        for b in ref_scn.alloc.table(ref_scn.seq_ids[r]):
            assert np.array_equal(kc[b].cpu().numpy().reshape(-1), ref_scn.pool.k[b].view(np.uint8).reshape(-1))
            assert np.array_equal(vc[b].cpu().numpy().reshape(-1), ref_scn.pool.v[b].view(np.uint8).reshape(-1))


def test_longest_context_at_table_capacity():
    """Sequences whose length fills the table exactly (ctx = max_blocks * T)."""
    w = W.scaled(W.get("long_mha_bf16"), num_seqs=2, num_q_heads=8, num_kv_heads=8, num_blocks=2100,
                 ctx_range=(32768, 32768))
    dev = PS.materialize(PS.plan(w), "cuda")
    assert dev.plan.max_blocks * w.block_size == 32768
    out = dev.step()
    torch.cuda.synchronize()
    ref_scn = OS.build(w, write_seqs=[0])
    ref = OA.paged_attention_decode(ref_scn.q_f64(), ref_scn.pool, ref_scn.tables, ref_scn.ctx,
                                    1.0 / math.sqrt(w.head_dim), seqs=[0])
    err = np.abs(out.double().cpu().numpy()[0] - ref[0])
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_prefill_full_size_sampled():
    """The chunked-prefill benchmark workload (16 chunks of 512 on contexts
    U[1024,4096], the tcgen05 kernel with ranked units), the whole batch on
    the GPU; the oracle recomputes the longest and the shortest sequence."""
    from oracle import prefill as OP
    w = W.get("qwen_prefill_bf16")
    dev = PS.materialize(PS.plan(w), "cuda")
    dev.copy_blocks()
    dev.write_step()
    ctx = dev.plan.ctx
    n = W.chunk_lens(w, ctx, w.prefill_chunk)
    qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = torch.cat([W.q_for_chunk(w, s, int(n[r])) for r, s in enumerate(dev.plan.seq_ids)])
    out = torch.full_like(q, float("nan"), device="cuda")
    pkv.pkv_attention_prefill(out, q.cuda(), dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                              torch.from_numpy(qs).cuda(), dev.desc, 1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert not np.isnan(got).any()
    rows = sorted({int(np.argmax(ctx)), int(np.argmin(ctx))})
    ref_scn = OS.build(w, write_seqs=rows)
    ref = OP.paged_attention_prefill(q.double().numpy(), ref_scn.pool, ref_scn.tables, ref_scn.ctx, qs,
                                     1.0 / math.sqrt(w.head_dim), seqs=rows)
    for r in rows:
        err = np.abs(got[qs[r]:qs[r + 1]] - ref[qs[r]:qs[r + 1]])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (r, err.max(), err.mean())


def test_prefill_one_long_prompt():
    """A whole 8,192-token prompt as one chunk (32 query-tile pairs, every
    causal diagonal), against the oracle on sampled query rows."""
    from oracle import prefill as OP
    w = W.scaled(W.get("qwen_prefill_bf16"), num_seqs=1, num_blocks=600, ctx_range=(8192, 8192),
                 seed=1399)
    dev = PS.materialize(PS.plan(w), "cuda")
    dev.copy_blocks()
    dev.write_step()
    n = int(dev.plan.ctx[0])
    qs = np.array([0, n], dtype=np.int32)
    q = W.q_for_chunk(w, dev.plan.seq_ids[0], n)
    out = torch.full_like(q, float("nan"), device="cuda")
    pkv.pkv_attention_prefill(out, q.cuda(), dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                              torch.from_numpy(qs).cuda(), dev.desc, 1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert not np.isnan(got).any()
    # the oracle on a few query rows: rows of a one-row chunk at position p are
    # the prefill rows of the whole prompt at p
    ref_scn = OS.build(w)
    for p in (0, 1, 127, 128, 4095, 8191):
        ref = OP.paged_attention_prefill(q[p:p + 1].double().numpy(), ref_scn.pool, ref_scn.tables,
                                         np.array([p + 1]), np.array([0, 1]), 1.0 / math.sqrt(w.head_dim))
        err = np.abs(got[p] - ref[0])
        assert err.max() <= 2e-2, (p, err.max())
