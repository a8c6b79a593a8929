"""Oracle pins: paged decode attention against brute force on contiguous
arrays, PyTorch's scaled_dot_product_attention, closed forms and the
invariants the pages state (values relocated, not transformed)."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import scenario as S
from oracle.allocator import BlockAllocator
from oracle.pool import PoolModel, bits_to_f64

TINY = W.get("tiny_fp32")
CASES = {
    "tiny_fp32": TINY,
    "tiny_gqa_fp32": W.scaled(TINY, num_q_heads=8, num_kv_heads=2, seed=77),
    "tiny_gqa_bf16": W.scaled(TINY, num_q_heads=6, num_kv_heads=2, head_dim=32, kv_dtype="bf16",
                              q_dtype="bf16", seed=78),
    "tiny_block4": W.scaled(TINY, block_size=4, num_blocks=160, seed=79),
}


def contiguous_kv(w, seq, ctx):
    """K, V of positions 0..ctx-1 straight from the generator (no pool)."""
    k0, v0 = W.kv_for_seq(w, seq, ctx - 1)
    k1, v1 = W.kv_for_seq(w, seq, 1, first_pos=ctx - 1)
    return (torch.cat([k0, k1]).double().numpy(), torch.cat([v0, v1]).double().numpy())


def brute_force(qv, K, V, scale):
    """Pure-Python softmax(q K^T scale) V."""
    n, d = len(K), len(qv)
    logits = [scale * sum(qv[i] * K[p][i] for i in range(d)) for p in range(n)]
    m = max(logits)
    wts = [math.exp(x - m) for x in logits]
    z = sum(wts)
    return [sum(wts[p] * V[p][i] for p in range(n)) / z for i in range(d)]


def oracle_out(scn):
    return A.paged_attention_decode(scn.q_f64(), scn.pool, scn.tables, scn.ctx,
                                    1.0 / math.sqrt(scn.w.head_dim))


def brute_error(scn):
    w = scn.w
    out = oracle_out(scn)
    g = w.num_q_heads // w.num_kv_heads
    q = scn.q_f64()
    err = 0.0
    for r, s in enumerate(scn.seq_ids):
        K, V = contiguous_kv(w, s, int(scn.ctx[r]))
        for j in range(w.num_q_heads):
            ref = brute_force(q[r, j].tolist(), K[:, j // g].tolist(), V[:, j // g].tolist(),
                              1.0 / math.sqrt(w.head_dim))
            err = max(err, float(np.max(np.abs(out[r, j] - np.array(ref)))))
    return err


@pytest.mark.parametrize("name", list(CASES))
def test_matches_brute_force_contiguous(name):
    assert brute_error(S.build(CASES[name])) < 1e-12


@pytest.mark.parametrize("name", list(CASES))
def test_matches_torch_sdpa(name):
    scn = S.build(CASES[name])
    w = scn.w
    out = oracle_out(scn)
    q = torch.from_numpy(scn.q_f64())
    for r, s in enumerate(scn.seq_ids):
        K, V = contiguous_kv(w, s, int(scn.ctx[r]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[r][None, :, None, :], torch.from_numpy(K).permute(1, 0, 2)[None],
            torch.from_numpy(V).permute(1, 0, 2)[None], scale=1.0 / math.sqrt(w.head_dim),
            enable_gqa=True)[0, :, 0, :].numpy()
        assert np.max(np.abs(out[r] - ref)) < 1e-12


def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(A, name, fn)


def test_pins_catch_a_dropped_scale(monkeypatch):
    orig = A.softmax_attention
    _planted(monkeypatch, "softmax_attention", lambda q, k, v, scale: orig(q, k, v, 1.0))
    assert brute_error(S.build(CASES["tiny_gqa_fp32"])) > 1e-6


def test_pins_catch_a_swapped_block_index(monkeypatch):
    def wrong_gather(cache, table, ctx, kv_head, block_size, kv_dtype, scale=1.0):
        p = np.arange(ctx)
        blk = np.asarray(table)[np.minimum(p % block_size, len(table) - 1)]
        rows = np.stack([cache[int(b)][kv_head, min(pp // block_size, block_size - 1)]
                         for b, pp in zip(blk, p)])
        return bits_to_f64(rows, kv_dtype, scale)
    _planted(monkeypatch, "gather_sequence", wrong_gather)
    assert brute_error(S.build(CASES["tiny_fp32"])) > 1e-6


def test_pins_catch_a_wrong_group_mapping(monkeypatch):
    w = CASES["tiny_gqa_fp32"]
    scn = S.build(w)
    good = oracle_out(scn)
    q = torch.from_numpy(scn.q_f64())
    # interleaved mapping j -> j % N_kv instead of contiguous groups
    def wrong(q_, pool, tables, ctx, scale, k_scale=1.0, v_scale=1.0, seqs=None):
        out = np.zeros_like(q_)
        for s in range(len(ctx)):
            for j in range(q_.shape[1]):
                h = j % pool.num_kv_heads
                k = A.gather_sequence(pool.k, tables[s], int(ctx[s]), h, pool.block_size, pool.kv_dtype)
                v = A.gather_sequence(pool.v, tables[s], int(ctx[s]), h, pool.block_size, pool.kv_dtype)
                out[s, j] = A.softmax_attention(q_[s, j], k, v, scale)
        return out
    bad = wrong(scn.q_f64(), scn.pool, scn.tables, scn.ctx, 1.0 / math.sqrt(w.head_dim))
    r, s = 0, scn.seq_ids[0]
    K, V = contiguous_kv(w, s, int(scn.ctx[r]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[r][None, :, None, :], torch.from_numpy(K).permute(1, 0, 2)[None],
        torch.from_numpy(V).permute(1, 0, 2)[None], scale=1.0 / math.sqrt(w.head_dim),
        enable_gqa=True)[0, :, 0, :].numpy()
    assert np.max(np.abs(good[r] - ref)) < 1e-12
    assert np.max(np.abs(bad[r] - ref)) > 1e-6


def test_physical_block_ids_do_not_change_the_output():
    """Values are relocated, not transformed: a different permutation of the
    pool gives bit-identical outputs."""
    a = S.build(W.scaled(TINY, shuffled_pool=False))
    b = S.build(TINY)
    assert a.tables != b.tables
    assert np.array_equal(oracle_out(a), oracle_out(b))


def _pool_with_tokens(alloc, pool, seq, k, v, n):
    slots, pairs = alloc.append(seq, n)
    pool.copy_blocks(pairs)
    kb = k.contiguous().view(torch.int32).numpy().view(np.uint32)
    vb = v.contiguous().view(torch.int32).numpy().view(np.uint32)
    pool.write(kb, vb, "f32", slots)


def test_shared_prefix_equals_private_copies():
    w = W.scaled(TINY, num_blocks=64)
    pk, pv = W.kv_for_seq(w, 100, 37)          # prefix, ends mid-block
    tails = [W.kv_for_seq(w, s, 11) for s in (0, 1)]
    outs = []
    for shared in (True, False):
        alloc = BlockAllocator(64, 16, W.free_order(w))
        pool = PoolModel(64, w.num_kv_heads, 16, w.head_dim, "f32", 0xFFFFFFFF)
        alloc.create(0)
        _pool_with_tokens(alloc, pool, 0, pk, pv, 37)
        if shared:
            alloc.fork(0, 1)
        else:
            alloc.create(1)
            _pool_with_tokens(alloc, pool, 1, pk, pv, 37)
        for s in (0, 1):
            _pool_with_tokens(alloc, pool, s, tails[s][0], tails[s][1], 11)
        q = np.stack([W.q_for_seq(w, s).double().numpy() for s in (0, 1)])
        outs.append(A.paged_attention_decode(q, pool, [alloc.table(0), alloc.table(1)], [48, 48], 0.125))
        if shared:  # two full prefix blocks shared; the partial one was copied
            assert alloc.table(0)[:2] == alloc.table(1)[:2] and alloc.table(0)[2] != alloc.table(1)[2]
    assert np.array_equal(outs[0], outs[1])


def _const_pool(k_rows, v_rows, block_size=4):
    n = len(k_rows)
    d = len(k_rows[0])
    nb = -(-n // block_size)
    pool = PoolModel(nb, 1, block_size, d, "f32", 0)
    kb = np.asarray(k_rows, dtype=np.float32).view(np.uint32)[:, None, :]
    vb = np.asarray(v_rows, dtype=np.float32).view(np.uint32)[:, None, :]
    pool.write(kb, vb, "f32", list(range(n)))
    return pool, [list(range(nb))]


def test_closed_form_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    n, d = 13, 8
    kr = np.tile(rng.standard_normal(d), (n, 1))
    vr = rng.standard_normal((n, d)).astype(np.float32)
    pool, tables = _const_pool(kr, vr)
    q = rng.standard_normal((1, 1, d))
    out = A.paged_attention_decode(q, pool, tables, [n], 0.3)
    assert np.allclose(out[0, 0], vr.astype(np.float64).mean(axis=0), atol=1e-14, rtol=0)


def test_closed_form_single_token_and_equal_values():
    rng = np.random.default_rng(2)
    d = 8
    kr = rng.standard_normal((9, d))
    vr = np.tile(rng.standard_normal(d).astype(np.float32), (9, 1))
    pool, tables = _const_pool(kr, vr)
    q = rng.standard_normal((1, 1, d)) * 5
    out = A.paged_attention_decode(q, pool, tables, [9], 1.0)
    assert np.allclose(out[0, 0], vr[0].astype(np.float64), atol=1e-14, rtol=0)
    vr2 = rng.standard_normal((9, d)).astype(np.float32)
    pool, tables = _const_pool(kr, vr2)
    out = A.paged_attention_decode(q, pool, tables, [1], 1.0)
    assert np.array_equal(out[0, 0], vr2[0].astype(np.float64))


def test_zero_context_gives_zero():
    pool, tables = _const_pool(np.ones((4, 8)), np.ones((4, 8)))
    out = A.paged_attention_decode(np.ones((1, 1, 8)), pool, tables, [0], 1.0)
    assert np.array_equal(out, np.zeros((1, 1, 8)))


def test_dominant_key_selects_its_value():
    """A key scaled far above the rest takes all the weight (the regime the
    long-context workload stresses with its scaled keys)."""
    rng = np.random.default_rng(3)
    d = 16
    kr = rng.standard_normal((20, d)) * 0.01
    q = rng.standard_normal(d)
    kr[7] = q * 50
    vr = rng.standard_normal((20, d)).astype(np.float32)
    pool, tables = _const_pool(kr, vr)
    out = A.paged_attention_decode(q[None, None], pool, tables, [20], 1.0)
    assert np.allclose(out[0, 0], vr[7].astype(np.float64), atol=1e-12)


def test_reading_an_unwritten_block_is_an_error():
    pool, tables = _const_pool(np.ones((4, 8)), np.ones((4, 8)))
    with pytest.raises(KeyError):
        A.paged_attention_decode(np.ones((1, 1, 8)), pool, [[0, 5]], [6], 1.0)
