"""Oracle pins: prefix caching in the block allocator, against the numbers and
rules the pages state (block-granular sharing: 992 of 1,000 tokens at block
size 32; a divergence inside a block loses the block; unrelated requests share
physical blocks; matched blocks are not recomputed) and invariants."""
import random

import pytest

from oracle.allocator import AllocError
from oracle.prefix_cache import PrefixCachingAllocator


def prompt(n, seed=0, vocab=50000):
    r = random.Random(seed)
    return [r.randrange(vocab) for _ in range(n)]


def run_prompt(a, seq, ids):
    """Create from the cache, append the rest with its ids; -> cached tokens."""
    hit = a.create_cached(seq, ids)
    a.append(seq, len(ids) - hit, ids[hit:])
    return hit


def test_shared_1000_token_prefix_reuses_992_at_block_32():
    """Foundry page, "Failure modes": block size 32, a shared 1,000-token
    prefix reuses at most 992 tokens."""
    a = PrefixCachingAllocator(200, 32)
    p = prompt(1000)
    assert run_prompt(a, 1, p) == 0
    assert run_prompt(a, 2, p) == 992
    assert a.table(2)[:31] == a.table(1)[:31]
    assert a.table(2)[31] != a.table(1)[31]      # the partial 32nd block is not shared


def test_divergence_inside_a_block_loses_that_block():
    a = PrefixCachingAllocator(200, 32)
    p = prompt(1000)
    run_prompt(a, 1, p)
    q = list(p)
    q[500] += 1                                  # inside block 15 (tokens 480..511)
    assert run_prompt(a, 2, q) == 480
    q2 = list(p)
    q2[479] += 1                                 # last token of block 14
    assert run_prompt(a, 3, q2) == 448


def test_unrelated_requests_share_physical_blocks_with_counts():
    a = PrefixCachingAllocator(64, 16)
    p = prompt(100, seed=3)
    run_prompt(a, 10, p)
    run_prompt(a, 11, p)
    run_prompt(a, 12, p + [7, 8, 9])
    shared = a.table(10)[:6]
    assert a.table(11)[:6] == shared and a.table(12)[:6] == shared
    assert all(a.block_refcount(b) == 3 for b in shared)
    a.free_seq(12)
    assert all(a.block_refcount(b) == 2 for b in shared)


def test_at_least_one_prompt_token_is_computed():
    a = PrefixCachingAllocator(200, 32)
    p = prompt(1024)                             # exactly 32 full blocks
    run_prompt(a, 1, p)
    assert run_prompt(a, 2, p) == 992            # 31 blocks, never all 32
    a2 = PrefixCachingAllocator(8, 16)
    run_prompt(a2, 1, prompt(16))
    assert a2.create_cached(2, prompt(16)) == 0  # a one-block prompt is always computed


def test_partial_blocks_are_never_published():
    """Prefix hashes are computed per filled block: 40 tokens at block 16
    publish 2 blocks."""
    a = PrefixCachingAllocator(16, 16)
    run_prompt(a, 1, prompt(40, seed=4))
    assert a.stats()[0] == 2
    assert run_prompt(a, 2, prompt(40, seed=4)) == 32


def test_freed_published_blocks_stay_reusable_until_evicted():
    a = PrefixCachingAllocator(8, 16, initial_free_order=list(range(8)))
    p = prompt(50, seed=5)                       # 3 full blocks + 2 tokens
    run_prompt(a, 1, p)
    t1 = a.table(1)
    a.free_seq(1)
    # the 3 published blocks wait, last block first; the partial one is free
    assert a.reusable() == [t1[2], t1[1], t1[0]]
    assert a.free_stack_top_first()[0] == t1[3]
    free_before = a.free_stack_top_first()
    assert run_prompt(a, 2, p) == 48
    assert a.table(2)[:3] == t1[:3]
    assert a.reusable() == []
    assert a.free_stack_top_first() == free_before[1:]   # only the tail block was popped


def test_eviction_takes_the_least_recently_freed_first():
    a = PrefixCachingAllocator(6, 16, initial_free_order=list(range(6)))
    pa, pb = prompt(64, seed=6), prompt(64, seed=7)   # 4 full blocks each
    run_prompt(a, 1, pa)                               # blocks 0..3, all four published
    a.free_seq(1)
    reuse = a.reusable()
    assert len(reuse) == 4
    run_prompt(a, 2, pb)          # needs 4 blocks: 2 from the stack, then 2 evicted
    assert a.stats()[3] == 2
    assert set(reuse[:2]) <= set(a.table(2))
    # pa's last two blocks are gone from the cache: a new request with pa
    # reuses only its first two blocks
    a.free_seq(2)
    assert a.create_cached(3, pa) == 32


def test_out_of_blocks_is_all_or_nothing():
    a = PrefixCachingAllocator(4, 16)
    run_prompt(a, 1, prompt(40, seed=8))
    state = (list(a.free), list(a.reuse), dict(a.key_to_entry))
    with pytest.raises(AllocError) as e:
        a.create(2)
        a.append(2, 33, prompt(33, seed=9))
    assert e.value.code == "OUT_OF_BLOCKS"
    assert (list(a.free), list(a.reuse), dict(a.key_to_entry)) == state


@pytest.mark.parametrize("seed", range(6))
def test_invariants_under_random_operations(seed):
    r = random.Random(seed)
    a = PrefixCachingAllocator(48, 4, initial_free_order=r.sample(range(48), 48))
    bases = [prompt(r.randrange(4, 30), seed=100 + i, vocab=5) for i in range(4)]
    live, nxt = [], 0
    for _ in range(400):
        op = r.random()
        try:
            if op < 0.35 or not live:
                ids = list(r.choice(bases))[: r.randrange(1, 31)] + prompt(r.randrange(0, 6),
                                                                           seed=r.random(), vocab=5)
                hit = a.create_cached(nxt, ids)
                assert hit % 4 == 0 and hit <= max(0, (len(ids) - 1) // 4 * 4)
                try:
                    a.append(nxt, len(ids) - hit, ids[hit:])
                except AllocError:
                    a.free_seq(nxt)
                    raise
                live.append(nxt)
                nxt += 1
            elif op < 0.6:
                s = r.choice(live)
                k = r.randrange(1, 6)
                ids = prompt(k, seed=r.random(), vocab=5) if r.random() < 0.5 else None
                a.append(s, k, ids)
            elif op < 0.7:
                a.fork(r.choice(live), nxt)
                live.append(nxt)
                nxt += 1
            else:
                s = live.pop(r.randrange(len(live)))
                a.free_seq(s)
        except AllocError as e:
            assert e.code == "OUT_OF_BLOCKS"
        # invariants
        refs = [0] * a.num_blocks
        for s in a.tables:
            for b in a.tables[s]:
                refs[b] += 1
        assert refs == a.refcount
        free, reuse = set(a.free), set(a.reuse)
        assert not free & reuse and len(free) == len(a.free) and len(reuse) == len(a.reuse)
        for b in range(a.num_blocks):
            assert (b in free or b in reuse) == (a.refcount[b] == 0)
            assert b not in reuse or a.block_entry[b] >= 0
        for e, b in a.entry_block.items():
            assert a.block_entry[b] == e
