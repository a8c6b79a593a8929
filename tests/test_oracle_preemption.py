"""Oracle pins: preemption by recompute and watermark admission, against the
behaviour the pages state (a dry pool preempts running sequences instead of
failing them; blocks are dropped and the sequence is re-prefilled later; under
sustained pressure a request is preempted and restarted several times) and
invariants."""
import random

import pytest

from oracle.allocator import AllocError, BlockAllocator
from oracle.prefix_cache import PrefixCachingAllocator
from oracle.preemption import admit, append_batch_preempt


def full_pool():
    """8 blocks of 4 tokens, 4 sequences holding 2 full blocks each."""
    a = BlockAllocator(8, 4)
    for s in range(4):
        a.create(s)
        a.append(s, 8)
    assert a.num_free() == 0
    return a


def test_dry_pool_preempts_the_lowest_priority_instead_of_failing():
    a = full_pool()
    t3 = a.table(3)
    slots, pairs, pre = append_batch_preempt(a, [0, 1, 2, 3])
    # seq 0 needs a block: seq 3 (lowest priority) goes, freeing 2 blocks for
    # seq 0 and seq 1; seq 2 then finds none and is itself the lowest left
    assert pre == [3, 2]
    assert slots[0] >= 0 and slots[1] >= 0 and slots[2] == slots[3] == -1
    assert pairs == []
    assert 2 not in a.tables and 3 not in a.tables
    assert a.table(0)[-1] in t3 and a.table(1)[-1] in t3
    assert a.context_len(0) == a.context_len(1) == 9


def test_no_preemption_when_blocks_suffice_and_only_as_many_as_needed():
    a = BlockAllocator(10, 4)
    for s in range(4):
        a.create(s)
        a.append(s, 8)
    slots, _, pre = append_batch_preempt(a, [0, 1, 2, 3])
    # 2 free blocks serve seqs 0 and 1; seq 2 then takes seq 3's blocks
    assert pre == [3] and slots[2] >= 0
    a2 = BlockAllocator(12, 4)
    for s in range(4):
        a2.create(s)
        a2.append(s, 8)
    slots, _, pre = append_batch_preempt(a2, [0, 1, 2, 3])
    assert pre == [] and all(x >= 0 for x in slots)


def test_unknown_or_duplicate_ids_change_nothing():
    a = full_pool()
    before = (list(a.free), dict(a.tables))
    with pytest.raises(AllocError):
        append_batch_preempt(a, [0, 9])
    with pytest.raises(AllocError):
        append_batch_preempt(a, [0, 0])
    assert (list(a.free), dict(a.tables)) == before


def test_watermark_admission():
    a = BlockAllocator(10, 4)
    admit(a, 0, 20, watermark=2)              # 5 blocks, 5 left >= 2
    with pytest.raises(AllocError) as e:
        admit(a, 1, 13, watermark=2)          # 4 blocks would leave 1 < 2
    assert e.value.code == "OUT_OF_BLOCKS" and 1 not in a.tables and a.num_free() == 5
    admit(a, 1, 12, watermark=2)              # 3 blocks leave exactly 2
    assert a.num_free() == 2


def serve(num_blocks, requests, watermark=1, block_size=4, caching=False, max_steps=10_000):
    """A recompute scheduler over the oracle: requests (prompt, output
    lengths) arrive in order; each step admits waiting requests in order
    (prompt plus tokens generated so far, above the watermark), then runs a
    decode step with preemption; a preempted request returns to the front of
    the waiting queue.  Returns per-request preemption counts and the
    allocator."""
    a = PrefixCachingAllocator(num_blocks, block_size) if caching else BlockAllocator(num_blocks, block_size)
    waiting = list(range(len(requests)))
    running, generated, preempts = [], [0] * len(requests), [0] * len(requests)
    tokens = {i: list(range(i * 10_000, i * 10_000 + requests[i][0])) for i in range(len(requests))}
    for _ in range(max_steps):
        while waiting:
            i = waiting[0]
            n = requests[i][0] + generated[i]
            try:
                if caching:
                    if -(-n // block_size) + watermark > a.num_free():
                        break
                    hit = a.create_cached(i, tokens[i][:n])
                    a.append(i, n - hit, tokens[i][hit:n])
                else:
                    admit(a, i, n, watermark)
            except AllocError:
                break
            running.append(waiting.pop(0))
        if not running and not waiting:
            break
        slots, _, pre = append_batch_preempt(a, running)
        for i, sl in zip(list(running), slots):
            if sl >= 0:
                generated[i] += 1
                tokens[i].append(i * 10_000 + 5_000 + generated[i])
        for i in pre:
            running.remove(i)
            preempts[i] += 1
        waiting = pre[::-1] + waiting          # the first preempted is served first
        for i in [i for i in running if generated[i] >= requests[i][1]]:
            running.remove(i)
            a.free_seq(i)
    assert not running and not waiting
    return preempts, a


def test_sustained_pressure_preempts_and_restarts_requests_several_times():
    r = random.Random(3)
    reqs = [(r.randrange(4, 20), r.randrange(20, 60)) for _ in range(12)]
    tight, _ = serve(24, reqs)
    roomy, _ = serve(400, reqs)
    assert max(tight) >= 2                   # restarted several times
    assert sum(roomy) == 0                   # enough blocks: no preemption at all


def test_recompute_finds_its_published_blocks_again():
    r = random.Random(4)
    reqs = [(r.randrange(20, 40), r.randrange(20, 40)) for _ in range(8)]
    preempts, a = serve(30, reqs, caching=True)
    assert sum(preempts) > 0
    assert a.stats()[2] > 0          # re-admissions were served partly from the cache


@pytest.mark.parametrize("seed", range(5))
def test_invariants_under_random_steps(seed):
    r = random.Random(seed)
    a = BlockAllocator(32, 4, initial_free_order=r.sample(range(32), 32))
    live, nxt = [], 0
    for _ in range(300):
        if r.random() < 0.3 or not live:
            try:
                admit(a, nxt, r.randrange(1, 20), r.randrange(0, 3))
                live.append(nxt)
            except AllocError as e:
                assert e.code == "OUT_OF_BLOCKS"
            nxt += 1
        elif r.random() < 0.15:
            a.fork(r.choice(live), nxt)
            live.append(nxt)
            nxt += 1
        else:
            batch = r.sample(live, len(live))
            before = {s: a.context_len(s) for s in batch}
            slots, _, pre = append_batch_preempt(a, batch)
            for s in pre:
                live.remove(s)
            # the preempted sequences are always a suffix of the priority order
            assert sorted(batch.index(s) for s in pre) == \
                list(range(len(batch) - len(pre), len(batch)))
            for i, s in enumerate(batch):
                if s in pre:
                    assert slots[i] == -1
                else:
                    assert slots[i] >= 0 and a.context_len(s) == before[s] + 1
        refs = [0] * a.num_blocks
        for s in a.tables:
            for b in a.tables[s]:
                refs[b] += 1
        assert refs == a.refcount
        assert sorted(a.free) == [b for b in range(a.num_blocks) if a.refcount[b] == 0]
