"""GPU parity of prefill attention (pkv_attention_prefill) against the CPU
oracle: max-abs 2e-2 and mean-abs 2e-3 for 16-bit caches.

The device state is the decode workloads' (each sequence's prior tokens and
the step token written through pkv_write); a sequence's chunk is its last
min(ctx, chunk) positions, whose K/V are therefore in the pool."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import prefill as OP
from oracle import scenario as OS

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3), "e4m3": (6e-2, None)}

CASES = {
    "qwen_small": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=8, num_blocks=600, ctx_range=(1, 1000)),
    "qwen_small_f16": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=6, num_blocks=500,
                               ctx_range=(1, 900), kv_dtype="f16", q_dtype="f16", seed=91),
    "mha_t32": W.scaled(W.get("long_mha_bf16"), num_seqs=3, num_q_heads=4, num_kv_heads=4,
                        num_blocks=200, ctx_range=(300, 1500), seed=94),
    "gqa16_d64": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=5, num_q_heads=32, num_kv_heads=2,
                          head_dim=64, num_blocks=300, ctx_range=(1, 800), block_size=32, seed=93),
    "fp8_small": W.scaled(W.get("fp8_churn"), num_seqs=6, num_blocks=1024, churn=300,
                          ctx_range=(1, 900)),
    "fp8_t32_qf16": W.scaled(W.get("fp8_churn"), num_seqs=4, num_blocks=512, churn=100,
                             ctx_range=(300, 1100), block_size=32, q_dtype="f16", seed=1398),
}


def scales_for(w):
    return W.fp8_scales(*W.kv_amax(w)) if w.kv_dtype == "e4m3" else {}


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


_STATE = {}


def state(name):
    """(device scenario, oracle scenario) of a case, built once."""
    if name not in _STATE:
        w = CASES[name]
        sc = scales_for(w)
        dev = PS.materialize(PS.plan(w), "cuda", sc)
        dev.copy_blocks()
        dev.write_step()
        torch.cuda.synchronize()
        _STATE[name] = (dev, OS.build(w, scales=sc))
    return _STATE[name]


def chunk_inputs(dev, n):
    """Packed queries of chunk lengths n (per batch row) and the row offsets."""
    w = dev.plan.w
    qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = torch.cat([W.q_for_chunk(w, s, int(n[r])) for r, s in enumerate(dev.plan.seq_ids)])
    return q, qs


def run_prefill(dev, q, qs, ctx=None, max_query_len=None):
    w = dev.plan.w
    out = torch.full_like(q, float("nan"), device="cuda")
    qd = q.to("cuda")
    ctx_t = dev.ctx if ctx is None else torch.from_numpy(np.asarray(ctx, dtype=np.int32)).cuda()
    pkv.pkv_attention_prefill(out, qd, dev.k_cache, dev.v_cache, dev.tables, ctx_t,
                              torch.from_numpy(qs).cuda(), dev.desc, 1.0 / math.sqrt(w.head_dim),
                              max_query_len=max_query_len, k_scale=dev.scales.get("k_scale", 1.0),
                              v_scale=dev.scales.get("v_scale", 1.0))
    torch.cuda.synchronize()
    return out


def oracle(scn, q, qs, ctx=None):
    return OP.paged_attention_prefill(q.double().numpy(), scn.pool, scn.tables,
                                      scn.ctx if ctx is None else ctx, qs,
                                      1.0 / math.sqrt(scn.w.head_dim),
                                      scn.scales.get("k_scale", 1.0), scn.scales.get("v_scale", 1.0))


def check(got, ref, kv_dtype="bf16"):
    g = got.double().cpu().numpy()
    assert not np.isnan(g).any(), "NaN in the GPU output"
    err = np.abs(g - ref)
    max_tol, mean_tol = TOL[kv_dtype]
    assert err.max() <= max_tol, f"max abs error {err.max():.3g}"
    if mean_tol is not None:
        assert err.mean() <= mean_tol, f"mean abs error {err.mean():.3g}"


@pytest.fixture(params=["auto", "mma_sync"])
def prefill_kernel(request):
    """Run a test with the default choice (tcgen05 UMMA for 16-bit caches with
    head_dim 128) and with the mma.sync kernel forced."""
    pkv.pkv_set_prefill_kernel(request.param)
    yield request.param
    pkv.pkv_set_prefill_kernel("auto")


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("chunk", [1, 37, 64, 200, 10 ** 6])
def test_prefill_matches_oracle(name, chunk, prefill_kernel):
    dev, scn = state(name)
    n = W.chunk_lens(dev.plan.w, dev.plan.ctx, chunk)
    q, qs = chunk_inputs(dev, n)
    check(run_prefill(dev, q, qs), oracle(scn, q, qs), dev.plan.w.kv_dtype)


@pytest.mark.parametrize("name", ["qwen_small", "qwen_small_f16", "mha_t32", "fp8_small"])
def test_tcgen05_and_mma_sync_kernels_agree(name):
    """The two prefill kernels compute the same attention (rounding apart),
    E4M3 caches included (widened to f16 in shared memory on tcgen05)."""
    dev, _ = state(name)
    n = W.chunk_lens(dev.plan.w, dev.plan.ctx, 300)
    q, qs = chunk_inputs(dev, n)
    outs = []
    for kind in ("tcgen05", "mma_sync"):
        pkv.pkv_set_prefill_kernel(kind)
        try:
            outs.append(run_prefill(dev, q, qs).double())
        finally:
            pkv.pkv_set_prefill_kernel("auto")
    err = (outs[0] - outs[1]).abs()
    assert not torch.isnan(outs[0]).any() and err.max().item() <= TOL[dev.plan.w.kv_dtype][0]


def test_tcgen05_choice_rejects_other_caches():
    dev, _ = state("gqa16_d64")
    n = W.chunk_lens(dev.plan.w, dev.plan.ctx, 10)
    q, qs = chunk_inputs(dev, n)
    pkv.pkv_set_prefill_kernel("tcgen05")
    try:
        with pytest.raises(pkv.PkvError):
            run_prefill(dev, q, qs)
    finally:
        pkv.pkv_set_prefill_kernel("auto")


@pytest.mark.parametrize("name", ["qwen_small", "gqa16_d64", "fp8_small"])
def test_one_token_chunks_match_decode_kernel(name):
    """A one-token chunk with the decode query is decode attention."""
    dev, _ = state(name)
    qs = np.arange(len(dev.plan.seq_ids) + 1, dtype=np.int32)
    pre = run_prefill(dev, dev.q.cpu(), qs)
    dec = dev.attend().clone()
    torch.cuda.synchronize()
    err = (pre.double() - dec.double()).abs()
    assert err.max().item() <= TOL[dev.plan.w.kv_dtype][0]


def test_empty_chunks_and_whole_prompts_mixed():
    dev, scn = state("qwen_small")
    ctx = dev.plan.ctx
    n = np.array([0 if r % 3 == 0 else (int(ctx[r]) if r % 3 == 1 else min(int(ctx[r]), 65))
                  for r in range(len(ctx))])
    q, qs = chunk_inputs(dev, n)
    got = run_prefill(dev, q, qs)
    check(got, oracle(scn, q, qs))


def test_invalid_chunk_gives_nan_rows_and_leaves_others():
    dev, scn = state("qwen_small")
    ctx = dev.plan.ctx.copy()
    n = np.minimum(ctx, 20)
    q, qs = chunk_inputs(dev, n)
    bad_ctx = ctx.copy()
    bad_ctx[2] = int(n[2]) - 1           # fewer positions than queries
    got = run_prefill(dev, q, qs, ctx=bad_ctx).double().cpu().numpy()
    assert np.isnan(got[qs[2]:qs[3]]).all()
    keep = np.ones(len(got), dtype=bool)
    keep[qs[2]:qs[3]] = False
    ref = oracle(scn, q, qs)
    assert np.abs(got[keep] - ref[keep]).max() <= TOL["bf16"][0]


def test_physical_blocks_do_not_change_the_output():
    """Tile boundaries depend only on logical positions: a different
    permutation of the pool gives bit-identical outputs."""
    w = CASES["qwen_small"]
    outs, tables = [], []
    for shuffled in (True, False):
        wv = W.scaled(w, shuffled_pool=shuffled)
        dev = PS.materialize(PS.plan(wv), "cuda")
        dev.copy_blocks()
        dev.write_step()
        n = W.chunk_lens(wv, dev.plan.ctx, 100)
        q, qs = chunk_inputs(dev, n)
        outs.append(run_prefill(dev, q, qs))
        tables.append(dev.plan.tables)
    assert not np.array_equal(tables[0], tables[1])
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_unsupported_cache_is_rejected():
    w = W.get("tiny_fp32")
    desc = pkv.kv_desc(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, "f32")
    kc, vc = pkv.empty_cache(desc, "cuda")
    q = torch.zeros(3, w.num_q_heads, w.head_dim, dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.pkv_attention_prefill(torch.empty_like(q), q, kc, vc,
                                  torch.zeros(2, 8, dtype=torch.int32, device="cuda"),
                                  torch.tensor([2, 1], dtype=torch.int32, device="cuda"),
                                  torch.tensor([0, 2, 3], dtype=torch.int32, device="cuda"),
                                  desc, 0.1)


@pytest.mark.parametrize("scale", [-0.06, 0.0])
def test_non_positive_softmax_scale(scale):
    """Any finite scale is attention's (the automatic choice sends scales <= 0
    to the mma.sync kernel)."""
    dev, scn = state("qwen_small")
    n = W.chunk_lens(dev.plan.w, dev.plan.ctx, 150)
    q, qs = chunk_inputs(dev, n)
    out = torch.full_like(q, float("nan"), device="cuda")
    pkv.pkv_attention_prefill(out, q.cuda(), dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                              torch.from_numpy(qs).cuda(), dev.desc, scale)
    torch.cuda.synchronize()
    ref = OP.paged_attention_prefill(q.double().numpy(), scn.pool, scn.tables, scn.ctx, qs, scale)
    check(out, ref)


def test_many_units_take_the_per_sequence_grid():
    """More than 256 (sequence, query-tile pair) units (here through a large
    max_query_len) launch the tcgen05 kernel on its (pair, head, sequence)
    grid instead of the ranked one; same results."""
    dev, scn = state("qwen_small")
    n = W.chunk_lens(dev.plan.w, dev.plan.ctx, 300)
    q, qs = chunk_inputs(dev, n)
    check(run_prefill(dev, q, qs, max_query_len=70_000), oracle(scn, q, qs))
