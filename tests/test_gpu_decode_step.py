"""pkv_decode_step (the step's slot write fused with decode attention) against
pkv_write + pkv_attention_decode on the same device state: the pool bytes and
the outputs are bit-identical, for every kernel choice and cache type; and
against the oracle."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import scenario as OS

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32": W.get("tiny_fp32"),
    "qwen_small": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=8, num_blocks=600, ctx_range=(1, 1000)),
    "prefix_small": W.scaled(W.get("prefix_fork_bf16"), num_seqs=16, num_blocks=256, prefix_len=96,
                             tail_range=(1, 60)),
    "fp8_small": W.scaled(W.get("fp8_churn"), num_seqs=12, num_blocks=2048, churn=500,
                          ctx_range=(1, 1500)),
    "gqa16_d64": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=5, num_q_heads=32, num_kv_heads=2,
                          head_dim=64, num_blocks=300, ctx_range=(1, 800), block_size=32, seed=93),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


def scales_for(w):
    return W.fp8_scales(*W.kv_amax(w)) if w.kv_dtype == "e4m3" else {}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_fused_step_equals_write_then_attend(name, kernel):
    w = CASES[name]
    if kernel != "auto" and w.kv_dtype == "f32":
        pytest.skip("the fp32 cache has one kernel")
    sc = scales_for(w)
    p = PS.plan(w)
    pkv.pkv_set_attention_kernel(kernel)
    try:
        a = PS.materialize(p, "cuda", sc, partition_tokens=0)
        a.copy_blocks()
        a.write_step()
        out_a = a.attend().clone()
        b = PS.materialize(p, "cuda", sc, partition_tokens=0)
        b.copy_blocks()
        out_b = b.decode_step().clone()
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_attention_kernel("auto")
    assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8))
    assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8))
    ia = out_a.view(torch.int16) if out_a.element_size() == 2 else out_a.view(torch.int32)
    ib = out_b.view(torch.int16) if out_b.element_size() == 2 else out_b.view(torch.int32)
    assert torch.equal(ia, ib)


@pytest.mark.parametrize("name", ["qwen_small", "fp8_small"])
def test_fused_step_matches_the_oracle(name):
    w = CASES[name]
    sc = scales_for(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc, partition_tokens=0)
    out = dev.step().double().cpu().numpy()
    torch.cuda.synchronize()
    scn = OS.build(w, scales=sc)
    ref = OA.paged_attention_decode(scn.q_f64(), scn.pool, scn.tables, scn.ctx,
                                    1.0 / math.sqrt(w.head_dim), sc.get("k_scale", 1.0),
                                    sc.get("v_scale", 1.0))
    err = np.abs(out - ref)
    tol = 6e-2 if w.kv_dtype == "e4m3" else 2e-2
    assert not np.isnan(out).any() and err.max() <= tol


@pytest.mark.parametrize("name", ["qwen_small", "prefix_small", "fp8_small"])
@pytest.mark.parametrize("shared", [False, True])
def test_prepared_step_equals_the_call(name, shared):
    """DeviceScenario.prepare_step (the library's Prepared calls: arguments
    checked once, launched on a raw stream handle) gives the same pool bytes
    and outputs, bit for bit, as the step through the plain calls."""
    w = CASES[name]
    plan = PS.plan(w)
    if shared and not plan.shared_prefix_blocks:
        pytest.skip("no shared prefix in this batch")
    dev = PS.materialize(plan, "cuda", scales_for(w), shared_prefix=shared)
    ref = dev.step().clone()
    k_ref, v_ref = dev.k_cache.clone(), dev.v_cache.clone()
    run = dev.prepare_step()
    dev.out.fill_(float("nan"))
    run(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(dev.out.view(torch.int16), ref.view(torch.int16))
    # (bytes: unwritten slots hold a NaN poison pattern)
    assert torch.equal(dev.k_cache.view(torch.uint8), k_ref.view(torch.uint8))
    assert torch.equal(dev.v_cache.view(torch.uint8), v_ref.view(torch.uint8))
