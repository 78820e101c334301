"""Pins of the CPU oracle to facts other than itself (no GPU).

* identity block table == contiguous attention computed by torch's
  scaled_dot_product_attention in fp64 (a library special case);
* permuting physical block ids together with their data leaves the output
  bit-identical (the block table is the only link between logical and physical);
* context length 1 returns V_0 exactly; scale 0 gives the mean of V; constant V
  rows return that row; identical K rows give the mean of V;
* a NumPy brute force over the six-dimensional pool array agrees to 1e-12;
* the worked block tables printed on the pages resolve tokens to the
  (physical block, offset) pairs worked out by hand from them;
* the append writes exactly the slot those tables name and nothing else.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from paged_kv_cache_239_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pool_np(pool_t):
    return W.as_oracle_array(pool_t)


def _to64(arr):
    return oracle.bf16_bits_to_f64(arr) if arr.dtype == np.uint16 else arr.astype(np.float64)


def _identity_workload(dtype, L, H, Hkv, D, B, lens, seed):
    """Sequence b owns physical blocks b*maxb .. b*maxb+maxb-1, in order."""
    lens = np.asarray(lens, dtype=np.int32)
    maxb = max(1, max(-(-int(n) // B) for n in lens))
    batch = len(lens)
    tables = np.full((batch, maxb), -1, dtype=np.int32)
    for b, n in enumerate(lens):
        nb = -(-int(n) // B)
        tables[b, :nb] = b * maxb + np.arange(nb)
    wl = W.Workload("identity", dtype, L, H, Hkv, D, B, lens, tables, batch * maxb,
                    1.0 / math.sqrt(D), seed)
    return wl


CASES = [
    ("f32", 2, 2, 2, 64, 16, [1, 15, 16, 17, 40]),
    ("bf16", 3, 8, 2, 64, 16, [5, 33, 64, 100]),
    ("bf16", 2, 4, 1, 128, 32, [31, 32, 33, 70]),
    ("f32", 1, 6, 3, 128, 16, [2, 47]),
]


@pytest.mark.parametrize("dtype,L,H,Hkv,D,B,lens", CASES)
def test_identity_table_equals_sdpa(oracle_lib, dtype, L, H, Hkv, D, B, lens):
    wl = _identity_workload(dtype, L, H, Hkv, D, B, lens, seed=11)
    pool_t = W.make_pool(wl)
    q_t = W.make_queries(wl, 1)[0]
    pool64 = pool_t.double()
    q64 = q_t.double()
    g = H // Hkv
    maxb = wl.max_blocks
    for layer in range(L):
        out = oracle.decode_attention(W.as_oracle_array(q_t), _pool_np(pool_t), layer,
                                      wl.block_tables, wl.context_lens, H, wl.scale)
        for b, n in enumerate(wl.context_lens):
            n = int(n)
            # contiguous cache of sequence b: its maxb blocks laid end to end
            seq = pool64[b * maxb:(b + 1) * maxb, :, layer]        # [maxb, 2, Hkv, B, D]
            k = seq[:, 0].permute(1, 0, 2, 3).reshape(Hkv, maxb * B, D)[:, :n]
            v = seq[:, 1].permute(1, 0, 2, 3).reshape(Hkv, maxb * B, D)[:, :n]
            k = k.repeat_interleave(g, dim=0).unsqueeze(0)
            v = v.repeat_interleave(g, dim=0).unsqueeze(0)
            qq = q64[b].unsqueeze(0).unsqueeze(2)                  # [1, H, 1, D]
            ref = torch.nn.functional.scaled_dot_product_attention(qq, k, v, scale=wl.scale)
            np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_permutation_invariance(oracle_lib, dtype):
    wl = W.custom("perm", dtype, 2, 8, 4, 64, 16, [3, 16, 29, 77, 130], seed=5, spare_blocks=7)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    rng = np.random.default_rng(17)
    perm = rng.permutation(wl.num_blocks)
    pool2 = np.empty_like(pool)
    pool2[perm] = pool                     # block i moves to id perm[i]
    tables2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    for layer in range(2):
        a = oracle.decode_attention(q, pool, layer, wl.block_tables, wl.context_lens, 8, wl.scale)
        b = oracle.decode_attention(q, pool2, layer, tables2, wl.context_lens, 8, wl.scale)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token_returns_v0(oracle_lib, dtype):
    wl = W.custom("one", dtype, 2, 4, 2, 64, 16, [1, 1, 1], seed=3, spare_blocks=4)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    p64 = _to64(pool)
    out = oracle.decode_attention(q, pool, 1, wl.block_tables, wl.context_lens, 4, 0.37)
    for b in range(3):
        for h in range(4):
            v0 = p64[wl.block_tables[b, 0], 1, 1, h // 2, 0]
            assert np.array_equal(out[b, h], v0)


def test_scale_zero_is_mean_of_v(oracle_lib):
    wl = W.custom("mean", "bf16", 1, 4, 2, 128, 32, [5, 32, 33, 97], seed=9)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    p64 = _to64(pool)
    g = oracle.gather_kv(pool, 0, wl.block_tables, wl.context_lens, 97)
    out = oracle.decode_attention(q, pool, 0, wl.block_tables, wl.context_lens, 4, 0.0)
    v64 = _to64(g[1])
    for b, n in enumerate(wl.context_lens):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], v64[b, :n, h // 2].mean(axis=0), atol=1e-13)
    assert p64.shape[0] == wl.num_blocks


def test_constant_v_rows_and_identical_k_rows(oracle_lib):
    wl = W.custom("const", "f32", 1, 2, 1, 64, 16, [23, 50], seed=21)
    pool = _pool_np(W.make_pool(wl)).copy()
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    c = np.linspace(-2, 2, 64).astype(np.float32)
    pool_cv = pool.copy()
    pool_cv[:, 1] = c                          # every V row equals c
    out = oracle.decode_attention(q, pool_cv, 0, wl.block_tables, wl.context_lens, 2, wl.scale)
    np.testing.assert_allclose(out, np.broadcast_to(c.astype(np.float64), out.shape), atol=1e-14)
    pool_ck = pool.copy()
    pool_ck[:, 0] = np.float32(0.25)           # every K row identical -> uniform weights
    out2 = oracle.decode_attention(q, pool_ck, 0, wl.block_tables, wl.context_lens, 2, wl.scale)
    _, v, _ = oracle.gather_kv(pool_ck, 0, wl.block_tables, wl.context_lens, 50)
    for b, n in enumerate(wl.context_lens):
        for h in range(2):
            np.testing.assert_allclose(out2[b, h], v[b, :n, 0].astype(np.float64).mean(0),
                                       atol=1e-13)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_brute_force_agreement(oracle_lib, seed):
    rng = np.random.default_rng(seed)
    H, Hkv = [(2, 2), (8, 2), (4, 4)][seed - 1]
    lens = rng.integers(0, 70, size=4)
    wl = W.custom("tiny", "bf16", 2, H, Hkv, 64, 16, lens, seed=seed, spare_blocks=3)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    for layer in range(2):
        a = oracle.decode_attention(q, pool, layer, wl.block_tables, wl.context_lens, H, wl.scale)
        b = brute.decode_attention(_to64(q), _to64(pool), layer, wl.block_tables,
                                   wl.context_lens, H, wl.scale)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_empty_sequence_is_zero(oracle_lib):
    wl = W.custom("empty", "f32", 1, 2, 2, 64, 16, [0, 5], seed=4, spare_blocks=2)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    out = oracle.decode_attention(q, pool, 0, wl.block_tables, wl.context_lens, 2, wl.scale)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out))


def test_oracle_rejects_out_of_range_ids(oracle_lib):
    wl = W.custom("bad", "f32", 1, 2, 2, 64, 16, [20], seed=4)
    pool = _pool_np(W.make_pool(wl))
    q = W.as_oracle_array(W.make_queries(wl, 1)[0])
    bad = wl.block_tables.copy()
    bad[0, 1] = wl.num_blocks
    with pytest.raises(ValueError):
        oracle.decode_attention(q, pool, 0, bad, wl.context_lens, 2, wl.scale)
    with pytest.raises(ValueError):
        oracle.decode_attention(q, pool, 0, wl.block_tables, [wl.max_blocks * 16 + 1], 2, 1.0)


def _golden_tables():
    with open(os.path.join(GOLDEN, "page_block_tables.json")) as f:
        return json.load(f)["tables"]


@pytest.mark.parametrize("entry", _golden_tables(), ids=lambda e: e["page"])
def test_page_worked_tables_resolve_as_drawn(oracle_lib, entry):
    B = entry["block_size"]
    nb = entry["min_pool_blocks"]
    table = np.array([entry["block_table"]], dtype=np.int32)
    n = len(entry["block_table"]) * B
    wl = W.Workload("golden", "f32", 1, 1, 1, 16, B, np.array([n], np.int32), table, nb, 1.0, 7)
    pool = _pool_np(W.make_pool(wl))
    k, v, mask = oracle.gather_kv(pool, 0, table, [n], n)
    assert mask.all()
    for t, page, off in entry["tokens"]:
        assert np.array_equal(k[0, t, 0], pool[page, 0, 0, 0, off])
        assert np.array_equal(v[0, t, 0], pool[page, 1, 0, 0, off])
    # decode over one token per logical block reads that block's first slot
    q = np.zeros((1, 1, 16), np.float32)
    for j, page in enumerate(entry["block_table"]):
        out = oracle.decode_attention(q, pool, 0, table[:, : j + 1], [j * B + 1], 1, 1.0)
        # uniform weights over tokens 0..j*B; the last one is page's slot 0
        _, vv, _ = oracle.gather_kv(pool, 0, table, [j * B + 1], j * B + 1)
        assert np.array_equal(vv[0, j * B, 0], pool[page, 1, 0, 0, 0])
        np.testing.assert_allclose(out[0, 0], vv[0, :, 0].astype(np.float64).mean(0), atol=1e-12)


@pytest.mark.parametrize("entry", _golden_tables(), ids=lambda e: e["page"])
def test_append_writes_the_drawn_slot_only(oracle_lib, entry):
    B = entry["block_size"]
    nb = entry["min_pool_blocks"]
    L, Hkv, D = 3, 2, 16
    table = np.array([entry["block_table"]], dtype=np.int32)
    for t, page, off in entry["tokens"]:
        pool = np.zeros((nb, 2, L, Hkv, B, D), np.float32)
        k = np.arange(1, Hkv * D + 1, dtype=np.float32).reshape(1, Hkv, D)
        v = -k
        oracle.write_kv(pool, 1, k, v, table, [t])
        assert np.array_equal(pool[page, 0, 1, :, off], k[0])
        assert np.array_equal(pool[page, 1, 1, :, off], v[0])
        assert np.count_nonzero(pool) == 2 * Hkv * D


def test_append_then_decode_uses_new_token(oracle_lib):
    """A token written at position n and a decode over n+1 tokens: with identical
    K rows the output is the mean of the old V rows and the new one."""
    wl = W.custom("app", "f32", 2, 2, 2, 64, 16, [15, 16], seed=8, steps=1)
    pool = _pool_np(W.make_pool(wl)).copy()
    pool[:, 0] = 1.0
    k = np.ones((2, 2, 64), np.float32)
    v = np.full((2, 2, 64), 3.5, np.float32)
    tables = wl.block_tables.copy()
    for b, n in enumerate(wl.context_lens):
        if n % 16 == 0:
            tables[b, n // 16] = wl.free_stack.pop()
    oracle.write_kv(pool, 1, k, v, tables, wl.context_lens)
    lens1 = wl.context_lens + 1
    q = np.zeros((2, 2, 64), np.float32)
    out = oracle.decode_attention(q, pool, 1, tables, lens1, 2, wl.scale)
    _, vv, _ = oracle.gather_kv(pool, 1, tables, lens1, int(lens1.max()))
    for b, n in enumerate(lens1):
        assert np.all(vv[b, n - 1] == 3.5)
        np.testing.assert_allclose(out[b], vv[b, :n].astype(np.float64).mean(0), atol=1e-12)


@pytest.mark.parametrize("dtype,Hkv,B,extra", [("bf16", 2, 16, 7), ("f32", 3, 32, 1),
                                               ("bf16", 1, 16, 40)])
def test_gather_matches_numpy_slicing_with_padding(oracle_lib, dtype, Hkv, B, extra):
    """The batched gather (mini-infer, "Zero-Copy Batched Attention Gather"; its
    listing stops after the call, so the output beyond each length is a reading:
    zero rows and mask 0) against NumPy advanced indexing of the six-dimensional
    pool array, with max_len past the longest context so every sequence has a
    padded tail.  An inverted mask, a padding that is not zeroed, a swapped KV
    head or K/V half, or a wrong layer or slot fails it."""
    lens = [0, 1, B - 1, B, B + 1, 3 * B + 5]
    wl = W.custom("gpad", dtype, 3, 2 * Hkv, Hkv, 64, B, lens, seed=31 + Hkv, spare_blocks=3,
                  interleave=True)
    pool = _pool_np(W.make_pool(wl))
    layer = 2
    T = int(max(lens)) + extra
    k, v, mask = oracle.gather_kv(pool, layer, wl.block_tables, wl.context_lens, T)
    assert k.shape == v.shape == (len(lens), T, Hkv, 64)
    assert mask.shape == (len(lens), T) and mask.dtype == bool
    for b, n in enumerate(lens):
        t = np.arange(n)
        blk = wl.block_tables[b, t // B]
        # advanced indices separated by a slice: result [n, Hkv, D]
        np.testing.assert_array_equal(k[b, :n], pool[blk, 0, layer, :, t % B, :])
        np.testing.assert_array_equal(v[b, :n], pool[blk, 1, layer, :, t % B, :])
        assert mask[b, :n].all() and not mask[b, n:].any()
        assert not k[b, n:].any() and not v[b, n:].any()
    # the padded region is genuinely present for every sequence
    assert (~mask).sum() == sum(T - n for n in lens)
