"""Oracle pins: block and pool sizing against the numbers the pages print."""
import json
import os

import pytest

from oracle import sizing

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sizing_examples.json")))


def test_block_bytes_worked_example():
    g = GOLD["block_bytes"]
    assert sizing.block_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["block_size"],
                              g["elem_bytes"]) == g["bytes"]


def test_block_bytes_fp8_is_half_of_fp16():
    g = GOLD["block_bytes"]
    assert 2 * sizing.block_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["block_size"], 1) \
        == g["bytes"]


def test_block_bytes_rejects_nonpositive():
    with pytest.raises(ValueError):
        sizing.block_bytes(28, 4, 128, 0, 2)


def test_pool_capacity_example():
    g = GOLD["pool_capacity"]
    n = sizing.num_blocks_for_budget(g["kv_budget_bytes"], g["block_bytes"])
    assert abs(n - g["approx_blocks"]) / g["approx_blocks"] < g["rel_tol"]
    assert abs(n * g["block_size"] - g["approx_tokens"]) / g["approx_tokens"] < g["rel_tol"]
    # whole blocks only: one more block would exceed the budget
    assert n * g["block_bytes"] <= g["kv_budget_bytes"] < (n + 1) * g["block_bytes"]


def test_contiguous_reservation_example():
    g = GOLD["contiguous_reservation"]
    assert sizing.contiguous_waste_tokens(g["reserved"], g["used"]) == g["empty"]


def test_internal_waste_fraction_example():
    g = GOLD["internal_waste_fraction"]
    frac = sizing.contiguous_waste_tokens(g["reserved"], g["used"]) / g["reserved"]
    assert abs(frac - g["approx_fraction"]) <= g["abs_tol"]


def test_lazy_allocation_example():
    g = GOLD["lazy_allocation"]
    assert sizing.blocks_for_tokens(g["tokens"], g["block_size"]) == g["blocks"]


def test_prefix_granularity_example():
    g = GOLD["prefix_granularity"]
    assert sizing.shareable_prefix_tokens(g["prefix_tokens"], g["block_size"]) == g["reused_tokens"]


@pytest.mark.parametrize("block_size", [1, 16, 32])
def test_paged_waste_bound_all_lengths(block_size):
    g = GOLD["waste_bound"]
    for n in range(0, 4 * block_size + 3):
        w = sizing.paged_waste_tokens(n, block_size)
        assert 0 <= w <= block_size - 1
        # capacity covers the tokens and one block fewer would not
        b = sizing.blocks_for_tokens(n, block_size)
        assert b * block_size >= n and (b - 1) * block_size < max(n, 1)
    assert max(sizing.paged_waste_tokens(n, g["block_size"]) for n in range(1, 200)) == g["max_waste_tokens"]
