"""The native allocator's preemption (pkv_batch_append_preempt) and watermark
admission (pkv_seq_admit) against the oracle, bit-exact on random streams,
with and without prefix caching.  Host only."""
import random

import pytest

import paged_kv_cache_137_gb300 as pkv
from oracle.allocator import AllocError, BlockAllocator
from oracle.prefix_cache import PrefixCachingAllocator
from oracle.preemption import admit, append_batch_preempt


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()


def both(fn_native, fn_oracle):
    try:
        rn = fn_native()
    except pkv.PkvError as e:
        rn = ("error", e.code)
    try:
        ro = fn_oracle()
    except AllocError as e:
        ro = ("error", e.code)
    return rn, ro


@pytest.mark.parametrize("caching", [False, True])
@pytest.mark.parametrize("seed", range(5))
def test_random_streams_match_the_oracle(seed, caching):
    r = random.Random(2000 + seed)
    nb, t = r.choice([(24, 4), (40, 8)])
    order = r.sample(range(nb), nb)
    n = pkv.Pool(nb, t, order)
    o = PrefixCachingAllocator(nb, t, order) if caching else BlockAllocator(nb, t, order)
    if caching:
        n.enable_prefix_cache()
    live, nxt, preempted_total = [], 0, 0
    for _ in range(300):
        u = r.random()
        if u < 0.3 or not live:
            k, wm = r.randrange(1, 4 * t), r.randrange(0, 3)
            rn, ro = both(lambda: list(n.seq_admit(nxt, k, wm)), lambda: admit(o, nxt, k, wm))
            assert rn == ro
            if isinstance(rn, list):
                live.append(nxt)
            nxt += 1
        elif u < 0.4:
            parent = r.choice(live)
            n.seq_fork(parent, nxt)
            o.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif u < 0.5:
            s = live.pop(r.randrange(len(live)))
            n.seq_free(s)
            o.free_seq(s)
        else:
            batch = r.sample(live, len(live))
            sn, cn, pn = n.batch_append_preempt(batch)
            so, co, po = append_batch_preempt(o, batch)
            assert list(sn) == so and [tuple(p) for p in cn] == [tuple(p) for p in co] and pn == po
            preempted_total += len(pn)
            for s in pn:
                live.remove(s)
        assert list(n.free_stack()) == o.free_stack_top_first()
        assert n.num_free_blocks() == o.num_free()
        for b in range(nb):
            assert n.block_refcount(b) == o.block_refcount(b)
        for s in live:
            tab, ln = n.seq_table(s)
            assert list(tab) == o.table(s) and ln == o.context_len(s)
    assert preempted_total > 0


def test_duplicate_or_unknown_ids_change_nothing():
    n = pkv.Pool(8, 4)
    n.seq_admit(0, 8)
    before = list(n.free_stack())
    for bad in ([0, 0], [0, 5]):
        with pytest.raises(pkv.PkvError):
            n.batch_append_preempt(bad)
    assert list(n.free_stack()) == before and n.seq_table(0)[1] == 8
