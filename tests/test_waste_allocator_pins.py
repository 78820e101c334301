"""Pins of the oracle's allocator and fragmentation arithmetic (no GPU).

The figures come from 'Paged KV-Cache Memory Management' (mini-infer): the
contiguous-reservation example of section 'The Problem', the last-block bound of
'Memory Waste Analysis', and the free-list semantics of its BlockPool
(``list(range(n))``, ``pop()`` from the end, ``append`` on free, MemoryError
when empty).
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import waste
from oracle.allocator import FreeBlockStack

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _figures():
    with open(os.path.join(GOLDEN, "page_waste_figures.json")) as f:
        return json.load(f)


def test_contiguous_example_matches_printed_percent():
    ex = _figures()["contiguous_example"]
    frac = waste.contiguous_waste_fraction(ex["reserved"], ex["used"])
    assert round(100 * frac, ex["printed_decimals"]) == ex["printed_percent"]


def test_paged_bound_at_printed_example():
    pb = _figures()["paged_bound"]
    bound = waste.paged_waste_bound(pb["n_tokens"], pb["block_size"])
    assert bound == pb["numerator"] / pb["n_tokens"]
    assert 100 * bound < pb["printed_upper_percent"]
    # every length from 400 tokens up stays under the printed figure
    for n in range(pb["n_tokens"], pb["n_tokens"] + 4 * pb["block_size"]):
        assert waste.paged_waste_fraction(n, pb["block_size"]) <= waste.paged_waste_bound(
            n, pb["block_size"]) < pb["printed_upper_percent"] / 100


@pytest.mark.parametrize("B", [8, 16, 32])
def test_waste_matches_slot_by_slot_simulation(B):
    """Grow a sequence token by token, taking a block whenever the last one is
    full, and count the unused slots; compare with the closed form and bound."""
    blocks = 0
    for n in range(1, 5 * B + 3):
        if (n - 1) % B == 0:
            blocks += 1
        unused = blocks * B - n
        w = waste.paged_waste_fraction(n, B)
        assert w == unused / n
        assert w <= waste.paged_waste_bound(n, B)
        assert (w == waste.paged_waste_bound(n, B)) == (n % B == 1 or B == 1)


def test_block_bytes_matches_tensor_size():
    # mini-infer BlockPool defaults: 24 layers, 2 KV heads, block 16, head_dim 64, bf16
    t = torch.zeros((1, 2, 24, 2, 16, 64), dtype=torch.bfloat16)
    assert waste.block_bytes(24, 2, 16, 64, 2) == t.numel() * t.element_size() == 196608


def test_free_stack_lifo_semantics():
    s = FreeBlockStack(5)
    ref = list(range(5))
    assert [s.allocate_block() for _ in range(2)] == [ref.pop(), ref.pop()] == [4, 3]
    s.free_block(4)
    assert s.allocate_block() == 4
    assert s.num_free() == 3


def test_free_stack_exhaustion_message():
    s = FreeBlockStack(2)
    s.allocate_block()
    s.allocate_block()
    with pytest.raises(MemoryError, match="Out of KV-Cache Physical Blocks"):
        s.allocate_block()


def test_free_stack_rejects_double_free_and_foreign_ids():
    s = FreeBlockStack(3)
    b = s.allocate_block()
    s.free_block(b)
    with pytest.raises(ValueError):
        s.free_block(b)
    with pytest.raises(ValueError):
        s.free_block(3)


def test_free_stack_seeded_order():
    s = FreeBlockStack(4)
    s.seed([2, 0, 3, 1])
    assert [s.allocate_block() for _ in range(4)] == [1, 3, 0, 2]
    with pytest.raises(ValueError):
        s.seed([0, 1, 2, 3])  # blocks in use


def test_random_ops_never_hand_out_a_block_twice():
    rng = np.random.default_rng(0)
    s = FreeBlockStack(16)
    held = set()
    for _ in range(2000):
        if held and (rng.random() < 0.45 or s.num_free() == 0):
            b = int(rng.choice(sorted(held)))
            s.free_block(b)
            held.remove(b)
        else:
            b = s.allocate_block()
            assert b not in held
            held.add(b)
        assert s.num_free() + len(held) == 16
