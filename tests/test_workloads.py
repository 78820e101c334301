"""The seeded workloads: shapes, distinct block ids, waste bound (no GPU)."""
import numpy as np
import pytest

from oracle import waste
from paged_kv_cache_239_gb300 import workloads as W


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_named_workload_tables_are_valid(cfg):
    wl = W.named(cfg)
    used = []
    for b, n in enumerate(wl.context_lens):
        nb = -(-int(n) // wl.block_size)
        row = wl.block_tables[b]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < wl.num_blocks)
        assert np.all(row[nb:] == -1)
        used.extend(int(x) for x in row[:nb])
        assert waste.paged_waste_fraction(int(n), wl.block_size) <= (wl.block_size - 1) / int(n)
    assert len(used) == len(set(used)), "a physical block is shared by two sequences"
    assert not set(used) & set(wl.free_stack)
    assert len(used) + len(wl.free_stack) == wl.num_blocks
    assert wl.num_heads % wl.num_kv_heads == 0


def test_named_workload_shapes():
    assert W.named(1).context_lens.tolist() == [17, 40]
    w2 = W.named(2)
    assert w2.pool_shape()[1:] == (2, 24, 2, 16, 64) and w2.batch == 32 and w2.group == 8
    assert 16 <= w2.context_lens.min() and w2.context_lens.max() <= 800
    w3 = W.named(3)
    assert w3.batch == 256 and w3.num_layers == 32 and w3.group == 4 and w3.head_dim == 128
    assert 128 <= w3.context_lens.min() and w3.context_lens.max() <= 4096
    w4 = W.named(4)
    assert w4.context_lens.tolist() == [32768, 65536, 100000, 131072] and w4.num_blocks == 10293
    w5 = W.named(5)
    assert w5.group == 1 and w5.steps == 64 and set([1, 31, 32, 33, 64, 1024]) <= set(
        w5.context_lens.tolist())
    # enough free blocks for 64 appended tokens per sequence
    extra = sum(-(-(int(n) + 64) // 32) - (-(-int(n) // 32)) for n in w5.context_lens)
    assert len(w5.free_stack) >= extra


def test_large_batch_tables_are_interleaved():
    wl = W.named(3)
    # round-robin pops: consecutive logical blocks of one sequence are far apart
    gaps = np.abs(np.diff(wl.block_tables[0, :16].astype(np.int64)))
    assert np.median(gaps) > 8


def test_generators_are_deterministic():
    wl = W.named(1)
    a = W.make_pool(wl)
    b = W.make_pool(wl)
    assert bool((a == b).all())
    assert W.named(2).context_lens.tolist() == W.named(2).context_lens.tolist()
