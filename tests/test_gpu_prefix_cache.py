"""Prefix caching end to end on the GPU: requests that reuse published blocks
write K/V only for their uncached positions ("that part of prefill is
skipped"), and decode attention through their tables, which share physical
blocks with earlier (finished) requests, matches the oracle; the native and
oracle allocators produce bit-identical tables along the way."""
import math
import random

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle.pool import PoolModel
from oracle.scenario import POISON, torch_bits
from oracle.prefix_cache import PrefixCachingAllocator

import paged_kv_cache_137_gb300 as pkv

pytestmark = pytest.mark.gpu

W0 = W.scaled(W.get("qwen_gqa_bf16"), num_seqs=6, num_blocks=160, seed=97)


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


def test_cached_prefixes_attend_like_the_oracle():
    w, t = W0, W0.block_size
    r = random.Random(7)
    system = [r.randrange(1000) for _ in range(200)]          # a shared preamble
    prompts = [system[: r.randrange(40, 200)] + [r.randrange(1000) for _ in range(r.randrange(1, 90))]
               for _ in range(w.num_seqs)]
    nat = pkv.Pool(w.num_blocks, t, W.free_order(w))
    nat.enable_prefix_cache()
    ora = PrefixCachingAllocator(w.num_blocks, t, W.free_order(w))
    desc = pkv.kv_desc(w.num_blocks, w.num_kv_heads, w.head_dim, t, w.kv_dtype)
    kc, vc = pkv.empty_cache(desc, "cuda", fill_byte=0xFF)
    pool = PoolModel(w.num_blocks, w.num_kv_heads, t, w.head_dim, w.kv_dtype, POISON[w.kv_dtype])
    written = 0
    live = []
    for i, ids in enumerate(prompts):
        hit = nat.seq_create_cached(i, ids)
        assert hit == ora.create_cached(i, ids)
        slots, _ = nat.seq_append_tokens(i, ids[hit:])
        assert list(slots) == ora.append(i, len(ids) - hit, ids[hit:])[0]
        # only the uncached positions are computed and written
        k, v = W.kv_for_seq(w, i, len(ids) - hit, first_pos=hit)
        pkv.pkv_write(kc, vc, k.cuda(), v.cuda(), torch.from_numpy(np.asarray(slots)).cuda(), desc)
        pool.write(torch_bits(k), torch_bits(v), w.src_dtype, slots)
        written += len(ids) - hit
        live.append(i)
        if i % 2 == 1:                       # finish every other request: its published
            nat.seq_free(live[0])            # blocks stay reusable
            ora.free_seq(live.pop(0))
    assert written < sum(len(p) for p in prompts)     # the preamble was reused
    assert nat.prefix_cache_stats()[2] > 0
    tables = [ora.table(s) for s in live]
    for s, tab in zip(live, tables):
        assert list(nat.seq_table(s)[0]) == tab
    ctx = np.array([ora.context_len(s) for s in live])
    max_blocks = max(len(x) for x in tables)
    tab_np = np.full((len(live), max_blocks), -1, dtype=np.int32)
    for row, tab in enumerate(tables):
        tab_np[row, :len(tab)] = tab
    q = torch.stack([W.q_for_seq(w, s) for s in live])
    out = torch.empty_like(q, device="cuda")
    ws = pkv.workspace_for(len(live), w.num_q_heads, max_blocks, desc, 0, "cuda")
    pkv.pkv_attention_decode(out, q.cuda(), kc, vc, torch.from_numpy(tab_np).cuda(),
                             torch.from_numpy(ctx.astype(np.int32)).cuda(), desc,
                             1.0 / math.sqrt(w.head_dim), workspace=ws)
    torch.cuda.synchronize()
    ref = OA.paged_attention_decode(q.double().numpy(), pool, tables, ctx, 1.0 / math.sqrt(w.head_dim))
    got = out.double().cpu().numpy()
    err = np.abs(got - ref)
    assert not np.isnan(got).any()
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
