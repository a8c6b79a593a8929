"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact: slot writes, block copies (the whole pool), tables and reference
counts.  Attention: max-abs 2e-2 and mean-abs 2e-3 for 16-bit caches, max-abs
1e-4 for fp32, max-abs 6e-2 for E4M3 (against the oracle on the dequantised
cache).
"""
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

TOL = {"f32": (1e-4, None), "f16": (2e-2, 2e-3), "bf16": (2e-2, 2e-3), "e4m3": (6e-2, None)}

SMALL = {
    "tiny_fp32": W.get("tiny_fp32"),
    "qwen_small": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=8, num_blocks=600, ctx_range=(1, 1000),
                           partition_tokens=256),
    "qwen_small_f16": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=6, num_blocks=500, ctx_range=(1, 900),
                               kv_dtype="f16", q_dtype="f16", seed=91),
    "prefix_small": W.scaled(W.get("prefix_fork_bf16"), num_seqs=16, num_blocks=256, prefix_len=96,
                             tail_range=(1, 60)),
    "long_small": W.scaled(W.get("long_mha_bf16"), num_seqs=2, num_q_heads=4, num_kv_heads=4,
                           num_blocks=200, ctx_range=(1500, 3000)),
    "fp8_small": W.scaled(W.get("fp8_churn"), num_seqs=12, num_blocks=2048, churn=500,
                          ctx_range=(1, 1500)),
    "gqa16_d64": W.scaled(W.get("qwen_gqa_bf16"), num_seqs=5, num_q_heads=32, num_kv_heads=2,
                          head_dim=64, num_blocks=300, ctx_range=(1, 800), block_size=32, seed=93),
}


def scales_for(w):
    return W.fp8_scales(*W.kv_amax(w)) if w.kv_dtype == "e4m3" else {}


def oracle_out(scn, rows=None):
    return OA.paged_attention_decode(scn.q_f64(), scn.pool, scn.tables, scn.ctx,
                                     1.0 / math.sqrt(scn.w.head_dim), scn.scales.get("k_scale", 1.0),
                                     scn.scales.get("v_scale", 1.0), seqs=rows)


def check_close(got, ref, kv_dtype, rows=None):
    rows = list(range(len(got))) if rows is None else rows
    err = np.abs(got[rows] - ref[rows])
    assert not np.isnan(got[rows]).any(), "NaN in the GPU output"
    max_tol, mean_tol = TOL[kv_dtype]
    assert err.max() <= max_tol, f"max abs error {err.max():.3g} > {max_tol}"
    if mean_tol is not None:
        assert err.mean() <= mean_tol, f"mean abs error {err.mean():.3g} > {mean_tol}"
    return err


def pool_bits(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def oracle_pool_bits(scn, which):
    dense = scn.pool.dense(which)
    return dense.view(np.uint8).reshape(-1)


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    assert torch.cuda.is_available()


@pytest.fixture(params=["simt", "tc"])
def kernel(request):
    """Run a test once per decode kernel (CUDA-core, tensor-core split)."""
    pkv.pkv_set_attention_kernel(request.param)
    yield request.param
    pkv.pkv_set_attention_kernel("auto")


def tc_covers(w):
    return w.kv_dtype != "f32" and w.num_q_heads // w.num_kv_heads <= 16 and \
        (w.head_dim == 128 or (w.head_dim == 64 and w.kv_dtype != "e4m3"))


@pytest.mark.parametrize("name", list(SMALL))
def test_step_matches_oracle(name, kernel):
    w = SMALL[name]
    if kernel == "tc" and not tc_covers(w):
        pytest.skip("the tensor-core kernel does not cover this cache")
    sc = scales_for(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc)
    out = dev.step()
    torch.cuda.synchronize()
    ref = OS.build(w, scales=sc)
    # pool bytes after copies + writes: bit-exact, unwritten slots keep the poison
    assert np.array_equal(pool_bits(dev.k_cache).reshape(-1), oracle_pool_bits(ref, "k"))
    assert np.array_equal(pool_bits(dev.v_cache).reshape(-1), oracle_pool_bits(ref, "v"))
    # block tables and reference counts from the native allocator
    for r, s in enumerate(ref.seq_ids):
        tab = ref.alloc.table(s)
        assert dev.plan.tables[r, :len(tab)].tolist() == tab
    for b in range(w.num_blocks):
        assert dev.plan.pool.block_refcount(b) == ref.alloc.block_refcount(b)
    check_close(out.double().cpu().numpy(), oracle_out(ref), w.kv_dtype)


@pytest.mark.parametrize("name", ["qwen_small", "long_small", "fp8_small"])
@pytest.mark.parametrize("partition", [0, 64, 128, 512, 4096])
def test_partition_sizes_agree_with_oracle(name, partition, kernel):
    w = SMALL[name]
    if partition % w.block_size:
        pytest.skip("partition must be a multiple of the block size")
    sc = scales_for(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc, partition_tokens=partition)
    out = dev.step()
    torch.cuda.synchronize()
    ref = OS.build(w, scales=sc)
    check_close(out.double().cpu().numpy(), oracle_out(ref), w.kv_dtype)


def test_physical_permutation_is_bit_identical(kernel):
    w = SMALL["qwen_small"]
    a = PS.materialize(PS.plan(W.scaled(w, shuffled_pool=False)), "cuda").step().clone()
    dev_b = PS.materialize(PS.plan(w), "cuda")
    b = dev_b.step()
    torch.cuda.synchronize()
    assert not np.array_equal(dev_b.plan.tables, PS.plan(W.scaled(w, shuffled_pool=False)).tables)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_equals_private_copies_bitwise(kernel):
    """A forked sequence reading shared prefix blocks gives the same bits as a
    sequence holding a private copy of the same prefix."""
    w = W.scaled(W.get("qwen_gqa_bf16"), num_blocks=64)
    desc = pkv.kv_desc(64, 4, 128, 16, "bf16")
    outs = []
    pk, pv = W.kv_for_seq(w, 100, 37)
    tails = [W.kv_for_seq(w, s, 12) for s in (0, 1)]
    q = torch.stack([W.q_for_seq(w, s) for s in (0, 1)]).cuda()
    for shared in (True, False):
        pool = pkv.Pool(64, 16, W.free_order(w))
        kc, vc = pkv.empty_cache(desc, "cuda", fill_byte=0xFF)

        def put(seq, k, v):
            slots, cow = pool.seq_append(seq, k.shape[0])
            pkv.pkv_copy_blocks([kc], [vc], cow, desc)
            pkv.pkv_write(kc, vc, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), desc)

        pool.seq_create(0)
        put(0, pk, pv)
        if shared:
            pool.seq_fork(0, 1)
        else:
            pool.seq_create(1)
            put(1, pk, pv)
        for s in (0, 1):
            put(s, *tails[s])
        tables, ctx = pool.block_tables([0, 1], 4)
        out = torch.empty_like(q)
        ws = pkv.workspace_for(2, 4, 4, desc)   # sized for the kernel chosen
        pkv.pkv_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                 torch.from_numpy(ctx).cuda(), desc, 1 / math.sqrt(128), workspace=ws)
        torch.cuda.synchronize()
        outs.append(out.view(torch.int16).cpu())
    assert torch.equal(outs[0], outs[1])


def _single_block_case(ctx_len, poison=True):
    desc = pkv.kv_desc(8, 2, 128, 16, "bf16")
    kc, vc = pkv.empty_cache(desc, "cuda", fill_byte=0xFF if poison else 0)
    g = torch.Generator().manual_seed(3)
    k = torch.randn(ctx_len, 2, 128, generator=g).bfloat16()
    v = torch.randn(ctx_len, 2, 128, generator=g).bfloat16()
    slots = torch.arange(3 * 16, 3 * 16 + ctx_len, dtype=torch.int64)
    pkv.pkv_write(kc, vc, k.cuda(), v.cuda(), slots.cuda(), desc)
    q = torch.randn(1, 4, 128, generator=g).bfloat16().cuda()
    tables = torch.tensor([[3, -1]], dtype=torch.int32).cuda()
    return desc, kc, vc, k, v, q, tables


def test_single_token_context_returns_its_value_exactly(kernel):
    desc, kc, vc, k, v, q, tables = _single_block_case(1)
    out = torch.empty_like(q)
    pkv.pkv_attention_decode(out, q, kc, vc, tables, torch.tensor([1], dtype=torch.int32).cuda(),
                             desc, 0.1, workspace=pkv.workspace_for(1, 4, 2, desc))
    torch.cuda.synchronize()
    expect = v[0].repeat_interleave(2, dim=0)  # heads 0,1 -> kv 0; 2,3 -> kv 1
    assert torch.equal(out[0].cpu(), expect)


def test_zero_context_gives_zero_and_poison_is_never_read(kernel):
    desc, kc, vc, k, v, q, tables = _single_block_case(5)
    out = torch.full_like(q, 7.0)
    pkv.pkv_attention_decode(out, q, kc, vc, tables, torch.tensor([0], dtype=torch.int32).cuda(),
                             desc, 0.1, workspace=pkv.workspace_for(1, 4, 2, desc))
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), torch.zeros_like(out.cpu()))
    pkv.pkv_attention_decode(out, q, kc, vc, tables, torch.tensor([5], dtype=torch.int32).cuda(),
                             desc, 0.1, workspace=pkv.workspace_for(1, 4, 2, desc))
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()   # slots 5..15 of the block hold NaN bits


def test_invalid_table_entry_or_length_gives_nan(kernel):
    """Invalid device inputs give NaN outputs and set their bit in the
    device error word, which the host reads and clears."""
    desc, kc, vc, k, v, q, tables = _single_block_case(16)
    pkv.pkv_device_status(clear=True)
    out = torch.zeros_like(q)
    bad = torch.tensor([[3, 99]], dtype=torch.int32).cuda()   # 99 >= num_blocks
    pkv.pkv_attention_decode(out, q, kc, vc, bad, torch.tensor([20], dtype=torch.int32).cuda(), desc, 0.1,
                             workspace=pkv.workspace_for(1, 4, 2, desc))
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    assert pkv.pkv_device_status(clear=True) == pkv.PKV_DEVICE_BAD_TABLE
    out.zero_()
    pkv.pkv_attention_decode(out, q, kc, vc, tables, torch.tensor([33], dtype=torch.int32).cuda(),
                             desc, 0.1, workspace=pkv.workspace_for(1, 4, 2, desc))   # longer than 2 blocks
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    assert pkv.pkv_device_status(clear=True) == pkv.PKV_DEVICE_BAD_LENGTH
    # valid inputs leave the word clear
    pkv.pkv_attention_decode(out, q, kc, vc, tables, torch.tensor([16], dtype=torch.int32).cuda(),
                             desc, 0.1, workspace=pkv.workspace_for(1, 4, 2, desc))
    assert pkv.pkv_device_status() == 0
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("which", ["tc"])
def test_stage_wait_give_up_sets_status_and_nan_then_recovers(which):
    """The decode kernel's failure path, run on purpose: with a stage-wait
    limit of 0 every CTA gives up at its first stage wait, still waits (with
    its own bounded limit) for the copies it has in flight, writes NaN and
    sets PKV_DEVICE_WAIT_TIMEOUT; split partials merge into NaN and the
    counters end at zero.  Afterwards the same call is correct."""
    w = SMALL["qwen_small"]
    pkv.pkv_set_attention_kernel(which)
    dev = PS.materialize(PS.plan(w), "cuda", partition_tokens=256)
    dev.copy_blocks()
    dev.write_step()
    pkv.pkv_device_status(clear=True)
    try:
        pkv.pkv_set_stage_wait_limit(0)
        out = dev.attend().clone()
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_stage_wait_limit(50_000_000)
        pkv.pkv_set_attention_kernel("auto")
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVICE_WAIT_TIMEOUT
    ctx = dev.plan.ctx
    assert torch.isnan(out[torch.from_numpy(ctx > 0)]).all()
    n = len(dev.plan.seq_ids) * w.num_kv_heads
    assert torch.count_nonzero(dev.workspace[: 4 * n]).item() == 0
    pkv.pkv_set_attention_kernel(which)
    try:
        out = dev.attend()
    finally:
        pkv.pkv_set_attention_kernel("auto")
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    check_close(out.double().cpu().numpy(), oracle_out(OS.build(w)), w.kv_dtype)


def test_write_skips_negative_and_out_of_pool_slots():
    desc = pkv.kv_desc(4, 1, 64, 16, "f32")
    kc, vc = pkv.empty_cache(desc, "cuda", fill_byte=0)
    k = torch.ones(3, 1, 64).cuda()
    slots = torch.tensor([-1, 4 * 16, 5], dtype=torch.int64).cuda()
    pkv.pkv_write(kc, vc, k, k, slots, desc)
    torch.cuda.synchronize()
    flat = kc.view(-1, 64).cpu()
    assert flat[5].eq(1).all() and flat.sum() == 64


def test_fp8_write_is_bit_exact_against_codec_for_all_bf16_values():
    """Every bf16 bit pattern through the E4M3 slot write, compared with the
    oracle's codec (same fp32 product, same rounding)."""
    from oracle import e4m3
    desc = pkv.kv_desc(4096, 1, 128, 16, "e4m3")
    kc, vc = pkv.empty_cache(desc, "cuda", fill_byte=0)
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).reshape(512, 1, 128)
    finite = torch.isfinite(x.float())
    x = torch.where(finite, x, torch.zeros_like(x))
    slots = torch.arange(512, dtype=torch.int64)
    inv = 0.37
    pkv.pkv_write(kc, vc, x.cuda(), x.cuda(), slots.cuda(), desc, inv, inv)
    torch.cuda.synchronize()
    got = kc.view(-1, 128)[:512].cpu().numpy().reshape(-1)
    expect = e4m3.quantize_fp32(x.float().numpy().reshape(-1), inv)
    assert np.array_equal(got, expect)


def test_copy_blocks_multi_layer_bit_exact():
    desc = pkv.kv_desc(32, 2, 64, 16, "bf16")
    layers = [pkv.empty_cache(desc, "cuda") for _ in range(3)]
    for kc, vc in layers:
        kc.view(torch.int16).random_(-32768, 32767)
        vc.view(torch.int16).random_(-32768, 32767)
    before = [(kc.clone(), vc.clone()) for kc, vc in layers]
    pairs = np.array([[3, 9], [17, 4], [31, 0]], dtype=np.int32)
    pkv.pkv_copy_blocks([l[0] for l in layers], [l[1] for l in layers], pairs, desc)
    torch.cuda.synchronize()
    for (kc, vc), (k0, v0) in zip(layers, before):
        ek, ev = k0.clone(), v0.clone()
        for s, d in pairs:
            ek[d] = k0[s]
            ev[d] = v0[s]
        # compare raw bits: random bf16 patterns include NaNs
        assert torch.equal(kc.view(torch.int16), ek.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), ev.view(torch.int16))


@pytest.mark.parametrize("name", ["qwen_small", "prefix_small", "fp8_small", "gqa16_d64"])
def test_kernels_agree(name):
    """The CUDA-core and tensor-core kernels on the same device state."""
    w = SMALL[name]
    dev = PS.materialize(PS.plan(w), "cuda", scales_for(w))
    dev.copy_blocks()
    dev.write_step()
    outs = []
    try:
        for k in ("simt", "tc"):
            pkv.pkv_set_attention_kernel(k)
            ws = pkv.workspace_for(len(dev.plan.seq_ids), w.num_q_heads, dev.plan.max_blocks, dev.desc,
                                   dev.partition)
            outs.append(dev.attend(workspace=ws).double().cpu().numpy().copy())
    finally:
        pkv.pkv_set_attention_kernel("auto")
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert np.abs(outs[0] - o).max() <= TOL[w.kv_dtype][0]


def test_split_counters_are_zero_after_a_call():
    """The fused split-K merge leaves its arrival counters at zero."""
    w = SMALL["long_small"]
    dev = PS.materialize(PS.plan(w), "cuda", partition_tokens=512)
    for _ in range(3):
        dev.step()
    torch.cuda.synchronize()
    n = len(dev.plan.seq_ids) * w.num_kv_heads
    assert torch.count_nonzero(dev.workspace[: 4 * n]).item() == 0


@pytest.mark.parametrize("name", ["qwen_small", "fp8_small", "gqa16_d64"])
def test_automatic_partition_with_edited_lengths(name, kernel):
    """The automatic partition with some lengths cut to 0, 1, 63, 64 and 65
    tokens, so that empty sequences, one-token sequences and tile edges sit
    between long ones."""
    w = SMALL[name]
    if kernel == "tc" and not tc_covers(w):
        pytest.skip("the tensor-core kernel does not cover this cache")
    sc = scales_for(w)
    dev = PS.materialize(PS.plan(w), "cuda", sc, partition_tokens=0)
    dev.copy_blocks()
    dev.write_step()
    ctx = dev.plan.ctx.copy()
    cut = {0: 0, 1: 1, 2: 63, 3: 64, 4: 65}
    for r, n in cut.items():
        if r < len(ctx):
            ctx[r] = min(n, ctx[r])
    dev.ctx.copy_(torch.from_numpy(ctx.astype(np.int32)))
    out = dev.attend(partition_tokens=0).double().cpu().numpy()
    torch.cuda.synchronize()
    ref_scn = OS.build(w, scales=sc)
    ref = OA.paged_attention_decode(ref_scn.q_f64(), ref_scn.pool, ref_scn.tables, ctx,
                                    1.0 / math.sqrt(w.head_dim), sc.get("k_scale", 1.0),
                                    sc.get("v_scale", 1.0))
    check_close(out, ref, w.kv_dtype)
    if ctx[0] == 0:
        assert np.all(out[0] == 0)


def test_batch_of_one_short_and_one_long_sequence():
    """A single short sequence (one tile) and a single long one (the
    automatic partition splits it over many CTAs)."""
    for ctx_range in [(40, 40), (30000, 30000)]:
        w = W.scaled(W.get("long_mha_bf16"), num_seqs=1, num_q_heads=8, num_kv_heads=1,
                     num_blocks=1000, ctx_range=ctx_range, partition_tokens=0, seed=97)
        dev = PS.materialize(PS.plan(w), "cuda")
        out = dev.step().double().cpu().numpy()
        torch.cuda.synchronize()
        ref_scn = OS.build(w)
        check_close(out, oracle_out(ref_scn), "bf16")
