"""The allocation-free decode entry point.

pkv_attention_decode_noalloc exists for callers that cannot allocate device
memory (a plug-in whose host runtime owns all device memory and passes only
inputs and outputs, or a serving loop that must not call cudaMalloc because it
can synchronise the device).  Its split-K scratch is a fixed array inside the
library.  These tests call it through the C ABI twice in a row, on different
workloads, and compare each result with the workspace entry point's, within
the tolerance of the other 16-bit parity tests.  This file runs last, so a
failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS

pytestmark = pytest.mark.gpu

CASES = [
    (W.scaled(W.get("qwen_gqa_bf16"), num_seqs=8, num_blocks=600, ctx_range=(1, 1000)), 256),
    (W.scaled(W.get("long_mha_bf16"), num_seqs=2, num_q_heads=4, num_kv_heads=4, num_blocks=200,
              ctx_range=(1500, 3000)), 512),
]


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    pkv.build()
    results = []
    for w, part in CASES:
        dev = PS.materialize(PS.plan(w), "cuda", partition_tokens=part)
        dev.copy_blocks()
        dev.write_step()
        need = pkv.pkv_attention_workspace_bytes(len(dev.plan.seq_ids), w.num_q_heads,
                                                 dev.plan.max_blocks, dev.desc, part)
        assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES   # the scratch is really used
        ref = dev.attend().clone()
        results.append((dev, part, ref))
    # two calls in a row on the shared scratch, each checked against the
    # workspace entry point on the same inputs
    for dev, part, ref in results:
        out = torch.full_like(dev.q, float("nan"))
        pkv.pkv_attention_decode_noalloc(out, dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                                         dev.desc, dev.softmax_scale, 1.0, 1.0, part)
        torch.cuda.synchronize()
        got, exp = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert not np.isnan(got).any()
        err = np.abs(got - exp)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_noalloc_rejects_sizes_beyond_its_scratch():
    pkv.build()
    desc = pkv.kv_desc(65536, 8, 128, 16, "bf16")
    need = pkv.pkv_attention_workspace_bytes(512, 64, 512, desc, 256)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    st = pkv.lib().pkv_attention_decode_noalloc(None, None, pkv.PKV_BF16, None, None, None, 512, None,
                                                512, 64, ctypes.byref(desc), 0.1, 1.0, 1.0, 256, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    assert b"scratch" in pkv.lib().pkv_last_error()
