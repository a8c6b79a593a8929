"""The native allocator's prefix caching (libpkv, C ABI) against the oracle,
bit-exact on random operation streams: tables, context lengths, counts, the
free stack, the reusable list (eviction order), cached-token counts, the
cache statistics and error codes.  Host only."""
import random

import numpy as np
import pytest

import paged_kv_cache_137_gb300 as pkv
from oracle.allocator import AllocError
from oracle.prefix_cache import PrefixCachingAllocator


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()


def both(fn_native, fn_oracle):
    """Run one operation on both; -> (result or error code) pairs."""
    try:
        rn = fn_native()
    except pkv.PkvError as e:
        rn = ("error", e.code)
    try:
        ro = fn_oracle()
    except AllocError as e:
        ro = ("error", e.code)
    return rn, ro


def same_state(n: pkv.Pool, o: PrefixCachingAllocator, live):
    assert list(n.free_stack()) == o.free_stack_top_first()
    assert list(n.reusable_blocks()) == o.reusable()
    assert n.num_free_blocks() == o.num_free()
    for b in range(o.num_blocks):
        assert n.block_refcount(b) == o.block_refcount(b)
    for s in live:
        tab, ln = n.seq_table(s)
        assert list(tab) == o.table(s) and ln == o.context_len(s)
    assert n.prefix_cache_stats() == o.stats()


@pytest.mark.parametrize("seed", range(24))
def test_random_streams_match_the_oracle(seed):
    r = random.Random(1000 + seed)
    nb, t = r.choice([(40, 4), (64, 16), (24, 8)])
    order = r.sample(range(nb), nb)
    n = pkv.Pool(nb, t, order)
    n.enable_prefix_cache()
    o = PrefixCachingAllocator(nb, t, order)
    bases = [[r.randrange(6) for _ in range(r.randrange(t, 6 * t))] for _ in range(3)]
    live, nxt = [], 0
    for step in range(300):
        op = r.random()
        if op < 0.35 or not live:
            ids = list(r.choice(bases))[: r.randrange(1, 6 * t)] + \
                [r.randrange(6) for _ in range(r.randrange(0, t))]
            rn, ro = both(lambda: n.seq_create_cached(nxt, ids), lambda: o.create_cached(nxt, ids))
            assert rn == ro
            if isinstance(rn, int):
                rest = ids[rn:]
                rn2, ro2 = both(lambda: [list(x) for x in n.seq_append_tokens(nxt, rest)][0],
                                lambda: o.append(nxt, len(rest), rest)[0])
                assert rn2 == ro2
                live.append(nxt)
            nxt += 1
        elif op < 0.55:
            s = r.choice(live)
            k = r.randrange(1, 2 * t)
            if r.random() < 0.5:
                ids = [r.randrange(6) for _ in range(k)]
                rn, ro = both(lambda: [list(x) for x in n.seq_append_tokens(s, ids)],
                              lambda: [list(x) for x in o.append(s, k, ids)])
            else:
                rn, ro = both(lambda: [list(x) for x in n.seq_append(s, k)],
                              lambda: [list(x) for x in o.append(s, k)])
            if isinstance(rn, list):
                rn = [rn[0], [list(p) for p in np.asarray(rn[1]).reshape(-1, 2)]]
                ro = [ro[0], [list(p) for p in ro[1]]]
            assert rn == ro, f"step {step}"
        elif op < 0.65:
            k = r.randrange(1, 5)
            # half the batches may repeat a sequence
            seqs = r.choices(live, k=k) if r.random() < 0.5 else r.sample(live, min(len(live), k))
            rn, ro = both(lambda: list(n.batch_append(seqs)[0]), lambda: o.append_batch(seqs, 1)[0])
            assert rn == ro
        elif op < 0.72:
            parent = r.choice(live)
            rn, ro = both(lambda: n.seq_fork(parent, nxt), lambda: o.fork(parent, nxt))
            assert rn == ro
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(r.randrange(len(live)))
            n.seq_free(s)
            o.free_seq(s)
        same_state(n, o, live)
    _, _, hits, evictions = o.stats()
    assert hits > 0 and evictions > 0   # the stream exercised reuse and eviction


def test_992_of_1000_at_block_32_through_the_c_abi():
    n = pkv.Pool(100, 32)
    n.enable_prefix_cache()
    ids = list(range(1000))
    assert n.seq_create_cached(1, ids) == 0
    n.seq_append_tokens(1, ids)
    assert n.seq_create_cached(2, ids) == 992
    assert list(n.seq_table(2)[0]) == list(n.seq_table(1)[0][:31])


def test_enable_needs_an_empty_pool_and_cached_calls_need_it():
    n = pkv.Pool(16, 16)
    with pytest.raises(pkv.PkvError):
        n.seq_create_cached(1, [1, 2, 3])
    n.seq_create(5)
    with pytest.raises(pkv.PkvError):
        n.enable_prefix_cache()
