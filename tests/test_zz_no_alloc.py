"""The allocation-free decode entry point.

pkv_attention_decode_noalloc exists for callers that cannot allocate device
memory (a plug-in whose host runtime owns all device memory and passes only
inputs and outputs, or a serving loop that must not call cudaMalloc because it
can synchronise the device).  Its split-K scratch is a fixed array inside the
library.  These tests call it through the C ABI twice in a row, on different
workloads, and compare each result with the workspace entry point's and with
the CPU oracle, within the tolerance of the other 16-bit parity tests; they
also check that the calls change neither PyTorch's allocations nor the
device's free memory.  This file runs last, so a failure here leaves every
other test already run.
"""
import ctypes
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

CASES = [
    (W.scaled(W.get("qwen_gqa_bf16"), num_seqs=8, num_blocks=600, ctx_range=(1, 1000)), 256),
    (W.scaled(W.get("long_mha_bf16"), num_seqs=2, num_q_heads=4, num_kv_heads=4, num_blocks=200,
              ctx_range=(1500, 3000)), 512),
    # the automatic partition (0): two long sequences are split over many CTAs
    (W.scaled(W.get("long_mha_bf16"), num_seqs=2, num_q_heads=8, num_kv_heads=8, num_blocks=800,
              ctx_range=(12000, 16000), seed=95), 0),
]


def oracle_out(w):
    scn = OS.build(w)
    return OA.paged_attention_decode(scn.q_f64(), scn.pool, scn.tables, scn.ctx,
                                     1.0 / math.sqrt(w.head_dim))


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
        results.append((w, dev, part, ref, torch.full_like(dev.q, float("nan"))))
    torch.cuda.synchronize()
    # the first call on the device looks up the scratch array's address
    w, dev, part, _, out = results[0]
    pkv.pkv_attention_decode_noalloc(out, dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                                     dev.desc, dev.softmax_scale, 1.0, 1.0, part)
    torch.cuda.synchronize()
    allocated, free = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    # calls in a row on the shared scratch, each checked against the workspace
    # entry point on the same inputs and against the oracle
    for w, dev, part, ref, out in results:
        out.fill_(float("nan"))
        pkv.pkv_attention_decode_noalloc(out, dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.ctx,
                                         dev.desc, dev.softmax_scale, 1.0, 1.0, part)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == allocated
        assert torch.cuda.mem_get_info()[0] == free
        # (read back through host copies: nothing on the device is allocated)
        got, exp = out.cpu().double().numpy(), ref.cpu().double().numpy()
        assert not np.isnan(got).any()
        err = np.abs(got - exp)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        err = np.abs(got - oracle_out(w))
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
