"""Oracle pins: prefill (multi-query, causal) attention through block tables,
against brute force on contiguous arrays, PyTorch's scaled_dot_product_attention
with an explicit mask and with is_causal, decode attention (a one-token chunk),
closed forms, and planted mistakes."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import prefill as P
from oracle import scenario as S
from oracle.pool import PoolModel

TINY = W.get("tiny_fp32")
CASES = {
    "tiny_fp32": TINY,
    "tiny_gqa_fp32": W.scaled(TINY, num_q_heads=8, num_kv_heads=2, seed=77),
    "tiny_gqa_bf16": W.scaled(TINY, num_q_heads=6, num_kv_heads=2, head_dim=32, kv_dtype="bf16",
                              q_dtype="bf16", seed=78),
    "tiny_block4": W.scaled(TINY, block_size=4, num_blocks=160, seed=79),
}


def prefill_inputs(scn, chunk):
    """Queries of each sequence's last min(ctx, chunk) positions, packed, and
    the row offsets."""
    w = scn.w
    n = W.chunk_lens(w, scn.ctx, chunk)
    qs = np.concatenate([[0], np.cumsum(n)])
    q = np.concatenate([W.q_for_chunk(w, s, int(n[r])).double().numpy()
                        for r, s in enumerate(scn.seq_ids)])
    return q, qs, n


def contiguous_kv(w, seq, ctx):
    k0, v0 = W.kv_for_seq(w, seq, ctx - 1)
    k1, v1 = W.kv_for_seq(w, seq, 1, first_pos=ctx - 1)
    return (torch.cat([k0, k1]).double().numpy(), torch.cat([v0, v1]).double().numpy())


def oracle_prefill(scn, q, qs):
    return P.paged_attention_prefill(q, scn.pool, scn.tables, scn.ctx, qs,
                                     1.0 / math.sqrt(scn.w.head_dim))


def brute_force(qv, K, V, scale, last):
    """Pure-Python attention of one query over positions 0..last."""
    d = len(qv)
    logits = [scale * sum(qv[i] * K[p][i] for i in range(d)) for p in range(last + 1)]
    m = max(logits)
    wts = [math.exp(x - m) for x in logits]
    z = sum(wts)
    return [sum(wts[p] * V[p][i] for p in range(last + 1)) / z for i in range(d)]


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("chunk", [1, 5, 200])
def test_matches_brute_force_contiguous(name, chunk):
    scn = S.build(CASES[name])
    w = scn.w
    q, qs, n = prefill_inputs(scn, chunk)
    out = oracle_prefill(scn, q, qs)
    g = w.num_q_heads // w.num_kv_heads
    err = 0.0
    for r, s in enumerate(scn.seq_ids[:2]):
        ctx = int(scn.ctx[r])
        K, V = contiguous_kv(w, s, ctx)
        for i in range(int(n[r])):
            last = ctx - int(n[r]) + i
            for j in range(w.num_q_heads):
                ref = brute_force(q[qs[r] + i, j].tolist(), K[:, j // g].tolist(),
                                  V[:, j // g].tolist(), 1.0 / math.sqrt(w.head_dim), last)
                err = max(err, float(np.max(np.abs(out[qs[r] + i, j] - np.array(ref)))))
    assert err < 1e-12


@pytest.mark.parametrize("name", list(CASES))
def test_matches_torch_sdpa_with_mask(name):
    scn = S.build(CASES[name])
    w = scn.w
    q, qs, n = prefill_inputs(scn, 37)
    out = oracle_prefill(scn, q, qs)
    for r, s in enumerate(scn.seq_ids):
        ctx, nr = int(scn.ctx[r]), int(n[r])
        K, V = contiguous_kv(w, s, ctx)
        mask = torch.zeros(nr, ctx, dtype=torch.bool)
        for i in range(nr):
            mask[i, : ctx - nr + i + 1] = True
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[qs[r]:qs[r + 1]]).permute(1, 0, 2)[None],
            torch.from_numpy(K).permute(1, 0, 2)[None], torch.from_numpy(V).permute(1, 0, 2)[None],
            attn_mask=mask, scale=1.0 / math.sqrt(w.head_dim), enable_gqa=True)[0].permute(1, 0, 2)
        assert np.max(np.abs(out[qs[r]:qs[r + 1]] - ref.numpy())) < 1e-12


def test_whole_prompt_matches_sdpa_is_causal():
    """A chunk covering the whole context is ordinary causal attention."""
    scn = S.build(CASES["tiny_gqa_fp32"])
    w = scn.w
    q, qs, n = prefill_inputs(scn, 10 ** 6)
    assert np.array_equal(n, scn.ctx)
    out = oracle_prefill(scn, q, qs)
    for r, s in enumerate(scn.seq_ids):
        K, V = contiguous_kv(w, s, int(scn.ctx[r]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[qs[r]:qs[r + 1]]).permute(1, 0, 2)[None],
            torch.from_numpy(K).permute(1, 0, 2)[None], torch.from_numpy(V).permute(1, 0, 2)[None],
            is_causal=True, scale=1.0 / math.sqrt(w.head_dim), enable_gqa=True)[0].permute(1, 0, 2)
        assert np.max(np.abs(out[qs[r]:qs[r + 1]] - ref.numpy())) < 1e-12


@pytest.mark.parametrize("name", list(CASES))
def test_one_token_chunk_is_decode(name):
    scn = S.build(CASES[name])
    q = scn.q_f64()
    qs = np.arange(len(scn.seq_ids) + 1)
    pre = oracle_prefill(scn, q, qs)
    dec = A.paged_attention_decode(q, scn.pool, scn.tables, scn.ctx,
                                   1.0 / math.sqrt(scn.w.head_dim))
    assert np.max(np.abs(pre - dec)) < 1e-13


def _const_pool(k_rows, v_rows, block_size=4):
    n, d = len(k_rows), len(k_rows[0])
    nb = -(-n // block_size)
    pool = PoolModel(nb, 1, block_size, d, "f32", 0)
    pool.write(np.asarray(k_rows, dtype=np.float32).view(np.uint32)[:, None, :],
               np.asarray(v_rows, dtype=np.float32).view(np.uint32)[:, None, :], "f32", list(range(n)))
    return pool, [list(range(nb))]


def test_closed_forms_equal_keys_and_first_position():
    """Equal keys: the query at position p gets the mean of V[0..p]; the
    query at position 0 gets v_0 whatever the keys."""
    rng = np.random.default_rng(5)
    n, d = 11, 8
    kr = np.tile(rng.standard_normal(d), (n, 1))
    vr = rng.standard_normal((n, d)).astype(np.float32)
    pool, tables = _const_pool(kr, vr)
    q = rng.standard_normal((n, 1, d))
    out = P.paged_attention_prefill(q, pool, tables, [n], [0, n], 0.7)
    v64 = vr.astype(np.float64)
    for p in range(n):
        assert np.allclose(out[p, 0], v64[: p + 1].mean(axis=0), atol=1e-14, rtol=0)
    kr2 = rng.standard_normal((n, d)) * 3
    pool2, tables2 = _const_pool(kr2, vr)
    out2 = P.paged_attention_prefill(q, pool2, tables2, [n], [0, n], 1.0)
    assert np.array_equal(out2[0, 0], v64[0])


def test_pins_catch_an_off_by_one_mask(monkeypatch):
    scn = S.build(CASES["tiny_fp32"])
    q, qs, _ = prefill_inputs(scn, 5)
    good = oracle_prefill(scn, q, qs)
    for wrong in (lambda f, nq, c: np.arange(c)[None, :] < f + np.arange(nq)[:, None],
                  lambda f, nq, c: np.arange(c)[None, :] <= f + 1 + np.arange(nq)[:, None]):
        monkeypatch.setattr(P, "causal_mask", wrong)
        bad = oracle_prefill(scn, q, qs)
        assert np.nanmax(np.abs(bad - good)) > 1e-6 or np.isnan(bad).any()


def test_physical_block_ids_do_not_change_the_output():
    a = S.build(W.scaled(TINY, shuffled_pool=False))
    b = S.build(TINY)
    assert a.tables != b.tables
    qa, qsa, _ = prefill_inputs(a, 9)
    qb, qsb, _ = prefill_inputs(b, 9)
    assert np.array_equal(qa, qb)
    assert np.array_equal(oracle_prefill(a, qa, qsa), oracle_prefill(b, qb, qsb))


def test_more_queries_than_context_is_rejected():
    scn = S.build(CASES["tiny_fp32"])
    n = int(scn.ctx[0]) + 1
    q = np.zeros((n, scn.w.num_q_heads, scn.w.head_dim))
    with pytest.raises(ValueError):
        P.paged_attention_prefill(q, scn.pool, scn.tables[:1], scn.ctx[:1], [0, n], 1.0)
