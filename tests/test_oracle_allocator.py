"""Oracle pins: the block allocator against the pages' invariants and examples."""
import copy
import json
import os
import random

import pytest

from oracle import sizing
from oracle.allocator import AllocError, BlockAllocator
from oracle.scenario import apply_churn

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sizing_examples.json")))


def check_invariants(a: BlockAllocator):
    """Structural facts the pages state, checked on any allocator state."""
    refs = [0] * a.num_blocks
    for seq, tab in a.tables.items():
        for b in tab:
            refs[b] += 1
        # lazy allocation: exactly the blocks the length needs, waste < T
        assert len(tab) == sizing.blocks_for_tokens(a.lens[seq], a.block_size)
        assert 0 <= len(tab) * a.block_size - a.lens[seq] <= a.block_size - 1
    # the count of a block is the number of tables that list it
    assert refs == a.refcount
    free = set(a.free)
    assert len(free) == len(a.free), "a block is on the free stack twice"
    for b in range(a.num_blocks):
        assert (b in free) == (refs[b] == 0), f"block {b} free and referenced, or leaked"
    assert sum(a.refcount) == sum(len(t) for t in a.tables.values())


def test_initial_order_top_first_and_default():
    a = BlockAllocator(4, 16, [2, 0, 3, 1])
    a.create(7)
    slots, _ = a.append(7, 40)
    assert a.table(7) == [2, 0, 3]
    assert slots[0] == 2 * 16 and slots[16] == 0 and slots[39] == 3 * 16 + 7
    b = BlockAllocator(3, 16)
    b.create(0)
    b.append(0, 17)
    assert b.table(0) == [0, 1]


def test_slot_arithmetic_by_position():
    a = BlockAllocator(8, 16, [5, 1, 6, 0, 2, 3, 4, 7])
    a.create(0)
    slots, _ = a.append(0, 50)
    tab = a.table(0)
    for p, s in enumerate(slots):
        assert s == tab[p // 16] * 16 + p % 16


def test_blocks_taken_only_when_previous_fills():
    a = BlockAllocator(16, 16)
    a.create(0)
    for n in range(1, 100):
        before = a.num_free()
        a.append(0, 1)
        opened = before - a.num_free()
        assert opened == (1 if (n - 1) % 16 == 0 else 0)
        check_invariants(a)


def test_lazy_allocation_example():
    g = GOLD["lazy_allocation"]
    a = BlockAllocator(64, g["block_size"])
    a.create(0)
    a.append(0, g["tokens"])
    assert len(a.table(0)) == g["blocks"]


def test_shared_prompt_refcount_example():
    g = GOLD["shared_prompt_refcount"]
    a = BlockAllocator(1024, g["block_size"])
    a.create(0)
    a.append(0, g["prompt_tokens"])
    free_before = a.num_free()
    for c in range(1, g["num_sequences"]):
        a.fork(0, c)
    assert a.num_free() == free_before, "fork copies the table, not memory"
    for b in a.table(0):
        assert a.block_refcount(b) == g["refcount"]
    check_invariants(a)


def test_copy_on_write_only_when_a_branch_writes():
    a = BlockAllocator(16, 16)
    a.create(0)
    a.append(0, 20)            # one full block, one partial (4 tokens)
    a.fork(0, 1)
    shared_full, shared_tail = a.table(0)
    assert a.block_refcount(shared_tail) == 2
    slots, pairs = a.append(1, 1)   # child writes into the shared partial block
    assert len(pairs) == 1 and pairs[0][0] == shared_tail
    new_tail = pairs[0][1]
    assert a.table(1) == [shared_full, new_tail]
    assert slots == [new_tail * 16 + 4]
    assert a.block_refcount(shared_tail) == 1 and a.block_refcount(new_tail) == 1
    slots, pairs = a.append(0, 1)   # parent is sole owner again: in place
    assert pairs == [] and slots == [shared_tail * 16 + 4]
    check_invariants(a)


def test_full_shared_block_is_never_copied():
    a = BlockAllocator(16, 16)
    a.create(0)
    a.append(0, 32)
    a.fork(0, 1)
    slots, pairs = a.append(1, 1)
    assert pairs == [] and len(a.table(1)) == 3 and a.table(1)[:2] == a.table(0)
    check_invariants(a)


def test_free_pushes_in_logical_order():
    a = BlockAllocator(8, 16, [3, 5, 1, 0, 2, 4, 6, 7])
    a.create(0)
    a.append(0, 40)
    assert a.table(0) == [3, 5, 1]
    a.free_seq(0)
    assert a.free_stack_top_first()[:3] == [1, 5, 3]
    assert a.num_free() == 8


def test_out_of_blocks_is_all_or_nothing():
    a = BlockAllocator(4, 16)
    a.create(0)
    a.append(0, 40)
    snap = copy.deepcopy(a.__dict__)
    with pytest.raises(AllocError) as e:
        a.append(0, 40)        # needs 3 more blocks, 1 free
    assert e.value.code == "OUT_OF_BLOCKS"
    assert a.__dict__ == snap
    a.create(1)
    a.create(2)
    snap = copy.deepcopy(a.__dict__)
    with pytest.raises(AllocError):
        a.append_batch([1, 2], 1)  # the first fits, the second does not
    assert a.__dict__ == snap


def test_unknown_and_duplicate_sequences():
    a = BlockAllocator(4, 16)
    with pytest.raises(AllocError) as e:
        a.append(9, 1)
    assert e.value.code == "UNKNOWN_SEQ"
    a.create(1)
    with pytest.raises(AllocError):
        a.create(1)
    with pytest.raises(AllocError):
        a.fork(1, 1)
    with pytest.raises(AllocError):
        BlockAllocator(3, 16, [0, 1, 1])


def test_any_free_block_serves_any_request_after_churn():
    """No external fragmentation: after a scrambling churn, a request that
    needs exactly all free blocks succeeds."""
    rnd = random.Random(5)
    coin = [rnd.random() for _ in range(2000)]
    pick = [rnd.random() for _ in range(2000)]
    a = BlockAllocator(300, 16, list(rnd.sample(range(300), 300)))
    apply_churn(a, coin, pick, 16)
    check_invariants(a)
    assert a.num_free() == 300
    a.create(0)
    a.append(0, 300 * 16)
    assert a.num_free() == 0
    check_invariants(a)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_invariants(seed):
    rnd = random.Random(seed)
    t = rnd.choice([1, 4, 16])
    a = BlockAllocator(64, t, rnd.sample(range(64), 64))
    live, next_id = [], 0
    for _ in range(600):
        op = rnd.random()
        try:
            if op < 0.15 or not live:
                a.create(next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.65:
                s = rnd.choice(live)
                n = rnd.randint(0, 3 * t)
                before = copy.deepcopy(a.__dict__)
                old_len = a.context_len(s)
                slots, pairs = a.append(s, n)
                # every written slot is in a block this sequence owns alone
                tab = a.table(s)
                for p, sl in zip(range(old_len, old_len + n), slots):
                    assert sl == tab[p // t] * t + p % t
                    assert a.block_refcount(sl // t) == 1
                # copies happen only for a shared partial block being written
                for src, dst in pairs:
                    assert old_len % t != 0 and before["refcount"][src] > 1
            elif op < 0.8:
                c = next_id
                a.fork(rnd.choice(live), c)
                live.append(c)
                next_id += 1
            else:
                s = live.pop(rnd.randrange(len(live)))
                a.free_seq(s)
        except AllocError as e:
            assert e.code == "OUT_OF_BLOCKS"
        check_invariants(a)
    for s in live:
        a.free_seq(s)
    assert a.num_free() == 64 and sum(a.refcount) == 0


def test_append_batch_matches_sequential_appends():
    a = BlockAllocator(64, 16, list(range(63, -1, -1)))
    for s in range(4):
        a.create(s)
        a.append(s, 5 + 9 * s)
    a.fork(2, 10)
    b = copy.deepcopy(a)
    sl, pr = a.append_batch([10, 0, 1, 2, 3], 1)
    sl2, pr2 = [], []
    for s in [10, 0, 1, 2, 3]:
        x, y = b.append(s, 1)
        sl2 += x
        pr2 += y
    assert (sl, pr) == (sl2, pr2) and a.__dict__ == b.__dict__
