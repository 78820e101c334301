"""Wide CTAs of the mma.sync kernel -- one CTA per (sequence, KV head, head
chunk) holding the whole context, its warps' results merged in shared memory
and written without a combine -- against the fp64 oracle: tables of the
largest size a wide CTA takes, ragged lengths with the edge cases (0, 1, B-1,
B, B+1, a full table), the fused append, and the one-wave boundary past which
the heuristic splits contexts again ("vllmini", "The CUDA Block Kernel")."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (TOL, GpuPool, device_tables, gpu_decode, max_abs_err, oracle_decode,
                         pool_in_layout)
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def wide_max_blocks(D):
    """Blocks per table a wide CTA takes: 16 warps x 4 at head_dim 64, 8 warps
    x 6 at 128.  Wide CTAs run while a call has between a third of the SMs
    and all of them as (sequence, KV head, head chunk) CTAs."""
    return 64 if D == 64 else 48


CASES = [(64, 16, 8), (64, 32, 16), (64, 16, 1), (64, 32, 24), (128, 16, 4), (128, 32, 16),
         (128, 32, 7), (128, 16, 3)]


def _lens(Bs, maxb, seed, batch=28):
    """Edge-case lengths, then random ones up to `batch` sequences (28 x 2 KV
    heads = 56 CTAs: more than a third of 152 SMs)."""
    rng = np.random.default_rng(seed)
    edge = [0, 1, Bs - 1, Bs, Bs + 1, maxb * Bs, maxb * Bs - 1]
    return edge + [int(x) for x in rng.integers(1, maxb * Bs + 1, size=batch - len(edge))]


@pytest.mark.parametrize("D,Bs,G", CASES)
def test_wide_whole_contexts_match_oracle(cuda_device, D, Bs, G):
    Hkv = 2
    maxb = wide_max_blocks(D)
    wl = W.custom("wide", "bf16", 2, Hkv * G, Hkv, D, Bs, _lens(Bs, maxb, D + Bs + G), seed=G + D,
                  spare_blocks=4, interleave=True, max_blocks=maxb)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TENSOR_CORES)   # (16 heads at 128: not tcgen05)
    # the heuristic holds each context in one CTA: no partials, no workspace
    assert B.pa_decode_partition_blocks(gp.h, wl.batch, wl.num_heads, maxb) == maxb
    assert B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, maxb, 0) == 0
    bt, ln = device_tables(wl, cuda_device)
    ref = oracle_decode(wl, pool, q, 1)
    for pb in (0, maxb, 4 * maxb):   # automatic, and explicit partitions covering the table
        out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln, partition_blocks=pb)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), pb
        assert max_abs_err(out, ref) <= TOL["bf16"], pb
    # empty contexts give zero vectors
    for b, n in enumerate(wl.context_lens):
        if n == 0:
            assert torch.count_nonzero(out[b]) == 0
    assert B.pa_get_status() == 0
    gp.close()


@pytest.mark.parametrize("D,Bs,G", [(64, 16, 8), (128, 32, 16), (128, 16, 4)])
def test_wide_fused_append_matches_oracle(cuda_device, D, Bs, G):
    """The new token's row is stored by the warp that copies its block, or by
    warp 0 when the block lies past the context."""
    Hkv = 2
    maxb = wide_max_blocks(D)
    lens = [0, 1, Bs - 1, Bs, 3 * Bs + 2, maxb * Bs - 1]      # positions of the new token
    lens += [int(x) for x in np.random.default_rng(D + G).integers(0, maxb * Bs, size=22)]
    wl = W.custom("wide_fused", "bf16", 2, Hkv * G, Hkv, D, Bs, lens, seed=D + G, steps=1,
                  spare_blocks=3, max_blocks=maxb)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    k, v = W.make_new_tokens(wl, 1)
    tables = wl.block_tables.copy()
    for b, n in enumerate(wl.context_lens):
        if n % Bs == 0:
            tables[b, n // Bs] = wl.free_stack.pop()
    gp = GpuPool(wl, pool.to(cuda_device))
    B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TENSOR_CORES)
    bt = torch.from_numpy(tables).to(cuda_device)
    pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
    lens1 = wl.context_lens + 1
    ln1 = torch.from_numpy(lens1).to(cuda_device)
    assert B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, maxb, 0) == 0
    out = torch.full((wl.batch, wl.num_heads, D), float("nan"), device=cuda_device)
    B.pa_write_kv_and_decode(out, q.to(cuda_device), gp.h, 1, k[0].to(cuda_device),
                             v[0].to(cuda_device), pos, bt, maxb, ln1, wl.batch, Bs,
                             wl.num_heads, Hkv, D, wl.scale, 0, None, 0)
    host = W.as_oracle_array(pool).copy()
    oracle.write_kv(host, 1, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                    wl.context_lens)
    ref = oracle.decode_attention(W.as_oracle_array(q), host, 1, tables, lens1, wl.num_heads,
                                  wl.scale)
    torch.cuda.synchronize()
    assert max_abs_err(out, ref) <= TOL["bf16"]
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    assert B.pa_get_status() == 0
    gp.close()


def test_wide_one_wave_boundary(cuda_device):
    """As many (sequence, KV head) CTAs as SMs, or a third of them, run wide;
    one more, or one fewer, and the heuristic splits the contexts again
    (partials and the combine).  All match the oracle, and so does a table one
    block longer than a wide CTA takes."""
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    D, Bs, G = 64, 16, 4
    maxb = 12
    third = -(-sms // 3)
    for batch, wide in ((sms, True), (sms + 1, False), (third, True), (third - 1, False)):
        rng = np.random.default_rng(batch)
        lens = [int(x) for x in rng.integers(0, maxb * Bs + 1, size=batch)]
        wl = W.custom("wave", "bf16", 1, G, 1, D, Bs, lens, seed=batch, max_blocks=maxb,
                      interleave=True)
        pool = W.make_pool(wl)
        q = W.make_queries(wl, 1)[0]
        gp = GpuPool(wl, pool.to(cuda_device))
        pb = B.pa_decode_partition_blocks(gp.h, batch, G, maxb)
        assert (pb == maxb) == wide, (batch, pb)
        assert (B.pa_decode_workspace_size(gp.h, batch, G, maxb, 0) == 0) == wide
        bt, ln = device_tables(wl, cuda_device)
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
        torch.cuda.synchronize()
        assert max_abs_err(out, oracle_decode(wl, pool, q, 0)) <= TOL["bf16"]
        gp.close()
    # a table one block longer than a wide CTA takes is split
    maxb = wide_max_blocks(128) + 1
    lens = [maxb * 16, 5, 700] + [int(x) for x in np.random.default_rng(5).integers(0, 700, 30)]
    wl = W.custom("long", "bf16", 1, 16, 2, 128, 16, lens, seed=5, max_blocks=maxb)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    assert B.pa_decode_partition_blocks(gp.h, wl.batch, 16, maxb) < maxb
    bt, ln = device_tables(wl, cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_decode(wl, pool, q, 0)) <= TOL["bf16"]
    assert B.pa_get_status() == 0
    gp.close()


@pytest.mark.parametrize("layout", ["separate", "layer_major"])
@pytest.mark.parametrize("D,Bs,G", [(64, 16, 8), (128, 32, 16), (128, 16, 5)])
def test_wide_strided_layouts_match_oracle(cuda_device, layout, D, Bs, G):
    """Separate K and V caches (one layer) and layer-major caches [L, n, Hkv,
    B, D]: a wide CTA's tensor maps take the caches' own strides.  The decode,
    then the fused append -- whose row lands bit-exactly where the oracle puts
    it in the same layout -- and the decode over the new token."""
    Hkv = 2
    H = Hkv * G
    maxb = wide_max_blocks(D)
    L = 1 if layout == "separate" else 3
    wl = W.custom("wide_strided", "bf16", L, H, Hkv, D, Bs, _lens(Bs, maxb - 1, 7 * D + G),
                  seed=3 * G + D, spare_blocks=3, interleave=True, max_blocks=maxb, steps=1)
    fused = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    (kc, vc), h = pool_in_layout(wl, fused, layout, cuda_device)
    try:
        B.pa_pool_set_decode_kernel(h, B.PA_DECODE_TENSOR_CORES)
        assert B.pa_decode_partition_blocks(h, wl.batch, H, maxb) == maxb
        assert B.pa_decode_workspace_size(h, wl.batch, H, maxb, 0) == 0
        layer = L - 1
        bt, ln = device_tables(wl, cuda_device)
        qd = q.to(cuda_device)
        ref = oracle.decode_attention(W.as_oracle_array(q), W.as_oracle_array(fused), layer,
                                      wl.block_tables, wl.context_lens, H, wl.scale)
        out = torch.full((wl.batch, H, D), float("nan"), device=cuda_device)
        B.pa_decode_attention_partitioned(out, qd, h, layer, bt, maxb, ln, wl.batch, Bs, H, Hkv,
                                          D, wl.scale, 0, None, 0)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref) <= TOL["bf16"], layout

        k, v = W.make_new_tokens(wl, 1)
        tables = wl.block_tables.copy()
        for b, n in enumerate(wl.context_lens):
            if n % Bs == 0:
                tables[b, n // Bs] = wl.free_stack.pop()
        lens1 = wl.context_lens + 1
        out = torch.full((wl.batch, H, D), float("nan"), device=cuda_device)
        B.pa_write_kv_and_decode(out, qd, h, layer, k[0].to(cuda_device), v[0].to(cuda_device),
                                 torch.from_numpy(wl.context_lens.copy()).to(cuda_device),
                                 torch.from_numpy(tables).to(cuda_device), maxb,
                                 torch.from_numpy(lens1).to(cuda_device), wl.batch, Bs, H, Hkv,
                                 D, wl.scale, 0, None, 0)
        host = W.as_oracle_array(fused).copy()
        oracle.write_kv(host, layer, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                        wl.context_lens)
        ref1 = oracle.decode_attention(W.as_oracle_array(q), host, layer, tables, lens1, H,
                                       wl.scale)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref1) <= TOL["bf16"], (layout, "fused")
        if layout == "separate":
            want_k, want_v = host[:, 0, 0], host[:, 1, 0]
        else:
            want_k = np.ascontiguousarray(host[:, 0].transpose(1, 0, 2, 3, 4))
            want_v = np.ascontiguousarray(host[:, 1].transpose(1, 0, 2, 3, 4))
        assert np.array_equal(W.as_oracle_array(kc), want_k)
        assert np.array_equal(W.as_oracle_array(vc), want_v)
        assert B.pa_get_status() == 0
    finally:
        B.pa_pool_destroy(h)
