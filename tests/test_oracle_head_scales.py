"""Oracle pins: E4M3 caches with one scale per KV head.

The pages fix only the one-byte element of an FP8 cache; the per-head variant
reads KV head h as e4m3 * scale[h] and stores fp32(x * inv[h]).  Pinned here
by properties that do not restate that formula:
* equal per-head scales are the per-tensor cache, byte for byte and output
  for output;
* multiplying KV head h's keys by 2^a_h and values by 2^b_h (and the queries
  of its group by 2^-a_h) changes no stored byte when the scales come from
  per-head maxima, and multiplies that group's outputs by exactly 2^b_h; a
  per-tensor scale does not have this property;
* each head's dequantised values lie within E4M3's rounding bound of the
  source at that head's own scale, even when the heads' magnitudes differ by
  2^40;
* prefill of one-token chunks is decode attention with the same scales.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import e4m3
from oracle.attention import paged_attention_decode
from oracle.pool import PoolModel, bits_to_f64
from oracle.prefill import paged_attention_prefill
from oracle.scenario import torch_bits

N_KV, T, D, G = 4, 16, 64, 3


def source(seed, n_tokens, gains_k=None, gains_v=None):
    """bf16 K, V [n_tokens, N_kv, D] (N(0,1), then head h times its gain in
    fp32, exact for powers of two) and their bits."""
    r = np.random.default_rng(seed)
    k = r.standard_normal((n_tokens, N_KV, D), dtype=np.float32)
    v = r.standard_normal((n_tokens, N_KV, D), dtype=np.float32)
    kb = torch.from_numpy(k).to(torch.bfloat16).float().numpy()
    vb = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    if gains_k is not None:
        kb = kb * np.asarray(gains_k, dtype=np.float32)[None, :, None]
        vb = vb * np.asarray(gains_v, dtype=np.float32)[None, :, None]
    return (torch.from_numpy(kb).to(torch.bfloat16), torch.from_numpy(vb).to(torch.bfloat16))


def head_amax(x):
    return x.float().abs().amax(dim=(0, 2)).double().numpy()


def build_pool(k, v, scales, seqs_ctx):
    """Write the tokens of each sequence into its own blocks (sequence s,
    position p at block s * 8 + p // T)."""
    pool = PoolModel(64, N_KV, T, D, "e4m3", 0x7F)
    tables, off = [], 0
    for s, c in enumerate(seqs_ctx):
        slots = [(s * 8 + p // T) * T + p % T for p in range(c)]
        pool.write(torch_bits(k[off:off + c]), torch_bits(v[off:off + c]), "bf16", slots,
                   scales["k_inv_scale"], scales["v_inv_scale"])
        tables.append([s * 8 + b for b in range(-(-c // T))])
        off += c
    return pool, tables


CTX = [37, 1, 70, 16]


def queries(seed, scale_rows=None):
    q = np.random.default_rng(seed).standard_normal((len(CTX), N_KV * G, D))
    q = torch.from_numpy(q).to(torch.bfloat16).double().numpy()
    if scale_rows is not None:
        q = q * np.repeat(np.asarray(scale_rows, dtype=np.float64), G)[None, :, None]
    return q


def test_equal_head_scales_are_the_per_tensor_cache():
    k, v = source(1, sum(CTX))
    sc = W.fp8_scales(float(head_amax(k).max()), float(head_amax(v).max()))
    sh = {n: np.full(N_KV, x, dtype=np.float32) for n, x in sc.items()}
    pa, tab = build_pool(k, v, sc, CTX)
    pb, _ = build_pool(k, v, sh, CTX)
    for b in pa.k:
        assert np.array_equal(pa.k[b], pb.k[b]) and np.array_equal(pa.v[b], pb.v[b])
    q = queries(2)
    oa = paged_attention_decode(q, pa, tab, CTX, 0.125, sc["k_scale"], sc["v_scale"])
    ob = paged_attention_decode(q, pb, tab, CTX, 0.125, sh["k_scale"], sh["v_scale"])
    assert np.array_equal(oa, ob)


def test_power_of_two_head_gains_change_no_byte_and_scale_outputs_exactly():
    a = np.array([0, -3, 5, -9])            # log2 gains of K per head
    b = np.array([2, 0, -6, 4])             # and of V
    k0, v0 = source(3, sum(CTX))
    k1, v1 = source(3, sum(CTX), np.exp2(a), np.exp2(b))
    s0 = W.fp8_scales(head_amax(k0), head_amax(v0))
    s1 = W.fp8_scales(head_amax(k1), head_amax(v1))
    p0, tab = build_pool(k0, v0, s0, CTX)
    p1, _ = build_pool(k1, v1, s1, CTX)
    for blk in p0.k:
        assert np.array_equal(p0.k[blk], p1.k[blk]) and np.array_equal(p0.v[blk], p1.v[blk])
    q0 = queries(4)
    q1 = queries(4, np.exp2(-a))
    o0 = paged_attention_decode(q0, p0, tab, CTX, 0.125, s0["k_scale"], s0["v_scale"])
    o1 = paged_attention_decode(q1, p1, tab, CTX, 0.125, s1["k_scale"], s1["v_scale"])
    want = o0 * np.repeat(np.exp2(b).astype(np.float64), G)[None, :, None]
    assert np.array_equal(o1, want)
    # one scale for the whole tensor: the small heads' bytes move
    t1 = W.fp8_scales(float(head_amax(k1).max()), float(head_amax(v1).max()))
    pt, _ = build_pool(k1, v1, t1, CTX)
    assert any(not np.array_equal(p0.k[blk], pt.k[blk]) for blk in p0.k)


def test_each_head_is_within_the_rounding_bound_of_its_own_scale():
    gains = np.exp2(-13.0 * np.arange(N_KV))            # 1 .. 2^-39
    k, v = source(5, 200, gains, gains)
    sh = W.fp8_scales(head_amax(k), head_amax(v))
    st = W.fp8_scales(float(head_amax(k).max()), float(head_amax(v).max()))
    x = k.float().numpy().astype(np.float64)
    for sc, per_head in ((sh, True), (st, False)):
        inv = np.asarray(sc["k_inv_scale"], dtype=np.float32)
        scale = np.asarray(sc["k_scale"], dtype=np.float32)
        inv3 = inv.reshape(1, -1, 1) if inv.ndim else inv
        bytes_ = e4m3.quantize_fp32(k.float().numpy(), inv3)
        for h in range(N_KV):
            s_h = float(scale[h]) if scale.ndim else float(scale)
            got = bits_to_f64(bytes_[:, h], "e4m3", s_h)
            err = np.abs(got - x[:, h])
            # normal E4M3: half an ulp of 3 mantissa bits (2^-4 relative);
            # subnormal: half the 2^-9 step; plus the fp32 product's rounding
            bound = 2.0 ** -4 * np.abs(x[:, h]) * (1 + 2.0 ** -20) + 2.0 ** -10 * s_h
            if per_head:
                assert (err <= bound).all(), h
                assert np.median(err / np.abs(x[:, h])) < 2.0 ** -5
            elif h == N_KV - 1:
                # the smallest head underflows the shared scale: all zeros
                assert (got == 0).all()


def test_one_token_prefill_chunks_are_decode_with_per_head_scales():
    k, v = source(6, sum(CTX), np.exp2([0, -2, -4, -6]), np.exp2([1, 0, -1, -2]))
    sh = W.fp8_scales(head_amax(k), head_amax(v))
    pool, tab = build_pool(k, v, sh, CTX)
    q = queries(7)
    dec = paged_attention_decode(q, pool, tab, CTX, 0.125, sh["k_scale"], sh["v_scale"])
    qs = np.arange(len(CTX) + 1)
    pre = paged_attention_prefill(q, pool, tab, CTX, qs, 0.125, sh["k_scale"], sh["v_scale"])
    assert np.array_equal(dec, pre)


def test_per_head_scales_need_one_value_per_head():
    k, v = source(8, 4)
    pool = PoolModel(8, N_KV, T, D, "e4m3", 0)
    with pytest.raises(ValueError):
        pool.write(torch_bits(k), torch_bits(v), "bf16", [0, 1, 2, 3], np.ones(N_KV - 1), 1.0)
