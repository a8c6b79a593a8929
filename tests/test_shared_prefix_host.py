"""Host side of the shared-prefix decode path (no GPU): the allocator's
shared-prefix count against brute force over the tables, and the workspace
the shared-prefix calls need."""
import random

import numpy as np
import pytest

import workloads as W

import paged_kv_cache_137_gb300 as pkv
from paged_kv_cache_137_gb300 import scenario as PS


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv.build()
    pkv.lib()


def brute_shared_prefix(pool, ids):
    """Leading entries equal in every table, below every sequence's last
    position (tables read one by one)."""
    if not ids:
        return 0
    tabs = [pool.seq_table(s) for s in ids]
    k = min((ln - 1) // pool.block_size if ln > 0 else 0 for _, ln in tabs)
    t0 = tabs[0][0]
    n = 0
    while n < k and all(int(t[n]) == int(t0[n]) for t, _ in tabs):
        n += 1
    return n


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_gqa_bf16", "prefix_fork_bf16"])
def test_workload_plans(name):
    p = PS.plan(W.get(name))
    assert p.shared_prefix_blocks == brute_shared_prefix(p.pool, p.seq_ids)
    if name == "prefix_fork_bf16":
        # the 1,024-token prompt of every fork: 64 blocks of 16
        assert p.shared_prefix_blocks == 64
    else:
        assert p.shared_prefix_blocks == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_fork_trees(seed):
    """Random prompts, forks, appends (with copy-on-write) and frees; the
    count equals brute force for random sub-batches after every step."""
    rng = random.Random(seed)
    t = rng.choice([16, 32])
    pool = pkv.Pool(4000, t)
    live, nxt = [], 0
    for _ in range(120):
        op = rng.random()
        if op < 0.25 or not live:
            pool.seq_create(nxt)
            pool.seq_append(nxt, rng.randint(1, 6 * t))
            live.append(nxt)
            nxt += 1
        elif op < 0.55:
            parent = rng.choice(live)
            pool.seq_fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.9:
            s = rng.choice(live)
            pool.seq_append(s, rng.randint(1, 2 * t))
        else:
            s = live.pop(rng.randrange(len(live)))
            pool.seq_free(s)
        if live:
            batch = rng.sample(live, rng.randint(1, len(live)))
            assert pool.shared_prefix_blocks(batch) == brute_shared_prefix(pool, batch)


def test_edge_cases():
    pool = pkv.Pool(64, 16)
    assert pool.shared_prefix_blocks([]) == 0
    pool.seq_create(1)
    assert pool.shared_prefix_blocks([1]) == 0            # empty sequence
    pool.seq_append(1, 33)
    assert pool.shared_prefix_blocks([1]) == 2            # blocks before position 32
    pool.seq_fork(1, 2)
    assert pool.shared_prefix_blocks([1, 2]) == 2
    pool.seq_append(2, 1)                                 # copy-on-write of block 2 only
    assert pool.shared_prefix_blocks([1, 2]) == 2
    pool.seq_create(3)
    pool.seq_append(3, 40)
    assert pool.shared_prefix_blocks([1, 3]) == 0         # a private prompt shares nothing
    with pytest.raises(pkv.PkvError) as e:
        pool.shared_prefix_blocks([1, 99])
    assert e.value.code == "UNKNOWN_SEQ"


def _align256(x):
    return (x + 255) // 256 * 256


def test_shared_prefix_workspace_layout():
    """The prefix-fork batch: two tail split slots (the automatic 512
    positions per split past the prefix for 16-bit caches at block size 16;
    the tails reach 97 * 16 - 1,024 = 528 positions) plus the prefix pass's
    key ranges (on 152 SMs the pass takes about a quarter of them: 8 KV heads
    x 4 row pairs = 32 row units, 38 / 32 -> one range of all 1,024 keys),
    laid out as the decode workspace with S = 2 + 1 slots and two more
    counters."""
    desc = pkv.kv_desc(8192, 8, 128, 16, "bf16")
    b, hq, max_blocks = 256, 32, 97
    s = 2 + 1
    n = b * hq * s
    # counters [B][N_kv], the decode grid's exit count and the tail queue's
    # claim counter, then the partials
    want = _align256(4 * (b * 8 + 2)) + 2 * _align256(4 * n) + _align256(4 * n * 128)
    assert pkv.pkv_shared_prefix_workspace_bytes(b, hq, max_blocks, desc, 64, 0) == want
    # never smaller than the plain call's (used where the pass does not run)
    for pfx in (0, 1, 10, 96, 97):
        assert pkv.pkv_shared_prefix_workspace_bytes(b, hq, max_blocks, desc, pfx, 512) >= \
            pkv.pkv_attention_workspace_bytes(b, hq, max_blocks, desc, 512)
    assert pkv.pkv_shared_prefix_workspace_bytes(b, hq, max_blocks, desc, 98, 0) == 0   # > max_blocks
    assert pkv.pkv_shared_prefix_workspace_bytes(b, hq, max_blocks, desc, -1, 0) == 0
