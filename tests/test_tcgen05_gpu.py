"""The tcgen05 decode kernel (GQA groups that are multiples of 16 on bf16 pools
with head_dim 128; the automatic choice for them) against the
oracle: ragged lengths around the 128-token tile, every partition size, chunked
groups, the fused append, many more work items than SMs (persistent CTAs),
stale values past the context, bad ids / lengths, and replays of a captured
graph."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W
from gpu_helpers import GpuPool, device_tables, gpu_decode, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu

TOL = 2e-3
LENS = [0, 1, 15, 16, 127, 128, 129, 255, 256, 700, 1500]


def _status_clear():
    torch.cuda.synchronize()
    B.pa_get_status()


@pytest.mark.parametrize("Hkv,H,Bs", [(1, 16, 16), (2, 32, 16), (1, 64, 32), (2, 128, 16),
                                       (1, 48, 16), (1, 96, 32), (1, 128, 16), (1, 192, 32),
                                       (1, 128, 32), (2, 256, 16), (1, 256, 32),
                                       (1, 80, 16), (2, 224, 32)])
def test_groups_match_oracle_every_partition(cuda_device, Hkv, H, Bs):
    wl = W.custom("tc", "bf16", 2, H, Hkv, 128, Bs, LENS, seed=H + Bs, spare_blocks=3,
                  interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    ref = oracle_decode(wl, pool, q, 1)
    _status_clear()
    try:
        for kind in (B.PA_DECODE_AUTO, B.PA_DECODE_TCGEN05):
            B.pa_pool_set_decode_kernel(gp.h, kind)
            for pb in (0, 1, 2, 8, 16, wl.max_blocks):
                out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln, partition_blocks=pb)
                err = max_abs_err(out, ref)
                assert err <= TOL, (kind, pb, err)
        # the mma.sync kernel serves the same shapes (as 16- or 8-head chunks)
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TENSOR_CORES)
        out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln)
        assert max_abs_err(out, ref) <= TOL
        torch.cuda.synchronize()
        assert B.pa_get_status() == 0
    finally:
        gp.close()


def test_tcgen05_refuses_other_shapes(cuda_device):
    for (H, Hkv, D) in [(8, 1, 128), (24, 1, 128), (32, 1, 64)]:
        wl = W.custom("tcno", "bf16", 1, H, Hkv, D, 16, [5, 40], seed=3)
        pool = W.make_pool(wl)
        gp = GpuPool(wl, pool.to(cuda_device))
        try:
            B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
            q = W.make_queries(wl, 1)[0].to(cuda_device)
            bt, ln = device_tables(wl, cuda_device)
            with pytest.raises(B.PagedAttnError) as e:
                gpu_decode(gp, q, 0, bt, ln)
            assert e.value.code == B.PA_ERR_UNSUPPORTED
        finally:
            gp.close()


@pytest.mark.parametrize("H,Bs,pb", [(32, 16, 0), (64, 32, 4), (16, 16, 1), (128, 16, 0),
                                     (128, 32, 0)])
def test_fused_append_matches_oracle(cuda_device, H, Bs, pb):
    wl = W.custom("tcapp", "bf16", 2, H, 1, 128, Bs, [0, 1, Bs - 1, Bs, 127, 128, 300, 511],
                  seed=11 + H, spare_blocks=4, interleave=True, steps=1)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        k, v = W.make_new_tokens(wl, 1)
        tables = wl.block_tables.copy()
        for b, n in enumerate(wl.context_lens):
            if n % Bs == 0:
                tables[b, n // Bs] = wl.free_stack.pop()
        btn = torch.from_numpy(tables).to(cuda_device)
        pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
        lens1 = wl.context_lens + 1
        out = torch.full((wl.batch, H, 128), float("nan"), device=cuda_device)
        need = B.pa_decode_workspace_size(gp.h, wl.batch, H, wl.max_blocks, pb)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
        _status_clear()
        B.pa_write_kv_and_decode(out, q.to(cuda_device), gp.h, 1, k[0].to(cuda_device),
                                 v[0].to(cuda_device), pos, btn, wl.max_blocks,
                                 torch.from_numpy(lens1).to(cuda_device), wl.batch, Bs, H, 1,
                                 128, wl.scale, pb, ws, need)
        host = W.as_oracle_array(pool).copy()
        oracle.write_kv(host, 1, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                        wl.context_lens)
        ref = oracle.decode_attention(W.as_oracle_array(q), host, 1, tables, lens1, H, wl.scale)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref) <= TOL
        assert np.array_equal(W.as_oracle_array(gp.t), host)
        assert B.pa_get_status() == 0
    finally:
        gp.close()


def test_many_more_items_than_sms(cuda_device):
    """Persistent CTAs walk the items in grid-stride order: 300 sequences x 2
    KV heads x up to 5 partitions, lengths ragged around the tile."""
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 600, size=300)]
    wl = W.custom("tcmany", "bf16", 1, 32, 2, 128, 16, lens, seed=78, interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        _status_clear()
        for pb in (0, 8):
            out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb)
            assert max_abs_err(out, ref) <= TOL, pb
        assert B.pa_get_status() == 0
    finally:
        gp.close()


@pytest.mark.parametrize("batch,H", [(200, 64), (160, 128), (200, 96)])
def test_combine_with_several_heads_per_warp(cuda_device, batch, H):
    """More (sequence, head group) pairs than decode CTAs, 64- or 48-head
    chunks: the combine then serves one record per decode CTA with 64 or 48
    heads each, more CTAs than fit the SMs at once with one head per warp, so
    each warp merges two heads (and the pairs cut once take the loads-first
    path)."""
    rng = np.random.default_rng(batch + H)
    lens = [int(x) for x in rng.integers(0, 1200, size=batch)]
    lens[:4] = [0, 1, 127, 129]
    wl = W.custom("tcrounds", "bf16", 1, H, 1, 128, 16, lens, seed=batch * 7 + H,
                  interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        assert B.pa_decode_kernel_choice(gp.h, H) == B.PA_DECODE_TCGEN05
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        _status_clear()
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
        assert torch.isfinite(out).all()
        assert max_abs_err(out, ref) <= TOL
        assert B.pa_get_status() == 0
    finally:
        gp.close()


def _poison_unused_rows(pool, wl):
    """NaN in every K/V row no sequence's context covers (free blocks and the
    rows past n in each last block)."""
    t = pool.clone()
    used = np.zeros(wl.num_blocks, bool)
    for b, n in enumerate(wl.context_lens):
        nblk = -(-int(n) // wl.block_size)
        for j in range(nblk):
            blk = int(wl.block_tables[b, j])
            used[blk] = True
            rows = min(wl.block_size, int(n) - j * wl.block_size)
            t[blk, :, :, :, rows:, :] = float("nan")
    for blk in np.nonzero(~used)[0]:
        t[int(blk)] = float("nan")
    return t


@pytest.mark.parametrize("H,Hkv,D,kind", [(32, 1, 128, "TCGEN05"), (128, 1, 128, "TCGEN05"),
                                         (16, 2, 128, "TENSOR_CORES"),
                                         (8, 2, 64, "TENSOR_CORES"), (8, 2, 64, "CUDA_CORES")])
def test_values_past_the_context_are_never_used(cuda_device, H, Hkv, D, kind):
    wl = W.custom("nan", "bf16", 1, H, Hkv, D, 16, [1, 7, 16, 100, 129, 250], seed=91,
                  spare_blocks=5, interleave=True)
    pool = _poison_unused_rows(W.make_pool(wl), wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, getattr(B, "PA_DECODE_" + kind))
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        assert np.isfinite(ref).all()
        for pb in (0, 1, wl.max_blocks):
            out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb)
            assert torch.isfinite(out).all(), pb
            assert max_abs_err(out, ref) <= TOL, pb
    finally:
        gp.close()


def test_bad_ids_and_lengths_flagged(cuda_device):
    wl = W.custom("tcbad", "bf16", 1, 32, 1, 128, 16, [300, 300, 300, 40], seed=5,
                  spare_blocks=2)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        tables = wl.block_tables.copy()
        tables[1, 3] = wl.num_blocks + 7
        tables[2, 12] = -1
        bt = torch.from_numpy(tables).to(cuda_device)
        lens = wl.context_lens.copy()
        lens[3] = wl.max_blocks * 16 + 1
        ln = torch.from_numpy(lens).to(cuda_device)
        _status_clear()
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln).cpu()
        st = B.pa_get_status()
        assert st & B.PA_STATUS_BAD_BLOCK_ID
        assert st & B.PA_STATUS_BAD_LENGTH
        assert not st & B.PA_STATUS_TIMEOUT
        assert torch.isfinite(out).all()
        ref = oracle_decode(wl, pool, q, 0)
        assert max_abs_err(out[0], ref[0]) <= TOL
        assert torch.all(out[3] == 0)
    finally:
        gp.close()


def test_graph_replays_match(cuda_device):
    wl = W.custom("tcgraph", "bf16", 1, 64, 1, 128, 16, [129, 1000, 3, 640], seed=21)
    pool = W.make_pool(wl)
    qs = W.make_queries(wl, 3)
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        bt, ln = device_tables(wl, cuda_device)
        qd = qs[0].to(cuda_device).clone()
        out = torch.zeros((wl.batch, 64, 128), device=cuda_device)
        need = B.pa_decode_workspace_size(gp.h, wl.batch, 64, wl.max_blocks, 2)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                B.pa_decode_attention_partitioned(out, qd, gp.h, 0, bt, wl.max_blocks, ln,
                                                  wl.batch, 16, 64, 1, 128, wl.scale, 2, ws,
                                                  need, s)
        torch.cuda.current_stream().wait_stream(s)
        for t in range(3):
            qd.copy_(qs[t].to(cuda_device))
            g.replay()
            torch.cuda.synchronize()
            assert max_abs_err(out, oracle_decode(wl, pool, qs[t], 0)) <= TOL, t
        assert B.pa_get_status() == 0
    finally:
        gp.close()


@pytest.mark.parametrize("lens,H,Hkv", [
    ([20000], 64, 1),                 # one context cut into a piece per CTA
    ([1], 64, 1),                     # one unit: a single CTA has work
    ([5000, 0, 3, 9000, 0], 128, 1),  # one 128-head chunk (heads on the rows), empty contexts
    ([5000, 0, 3, 9000, 0], 192, 1),  # three 64-head chunks, empty contexts
    ([700, 1500, 0, 129, 2047], 112, 1),  # 112 heads in one 128-head chunk (16 rows dropped)
    ([700, 1500, 0, 129, 2047], 48, 1),   # three 16-head chunks
    ([33000, 17, 128], 32, 2),        # long + short, two KV heads
])
def test_equal_tile_shares_split_anywhere(cuda_device, lens, H, Hkv):
    """Every CTA takes an equal run of 128-token tiles in (sequence, head
    group, tile) order, so contexts are cut at arbitrary tiles and merged by
    the combine; the result must not depend on where the cuts fall."""
    wl = W.custom("tcshare", "bf16", 1, H, Hkv, 128, 16, lens, seed=sum(lens) % 997 + H,
                  spare_blocks=2, interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        sizes = {B.pa_decode_workspace_size(gp.h, wl.batch, H, wl.max_blocks, pb)
                 for pb in (0, 1, wl.max_blocks)}
        assert len(sizes) == 1, sizes   # partition_blocks does not apply to it
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        _status_clear()
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
        assert max_abs_err(out, ref) <= TOL
        assert B.pa_get_status() == 0
    finally:
        gp.close()


def test_workspace_reused_across_calls_and_checked(cuda_device):
    """The per-CTA partial slots and the pair descriptors need no clearing: a
    workspace left by a call with other lengths (more pieces, other cuts) gives
    the same results; a workspace one byte short is refused before launch."""
    lens_a = [20000, 3, 0, 5000]
    lens_b = [129, 7000, 1, 0, 16000, 640]
    H = 64
    wl = W.custom("tcreuse", "bf16", 1, H, 1, 128, 16, lens_a + lens_b, seed=404,
                  spare_blocks=2, interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TCGEN05)
        need = B.pa_decode_workspace_size(gp.h, wl.batch, H, wl.max_blocks, 0)
        assert need > 0
        ws = torch.full((need,), 0xA5, dtype=torch.uint8, device=cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        na = len(lens_a)
        # first call: the first sequences only (same tables), then all of them
        tables = torch.from_numpy(wl.block_tables).to(cuda_device)
        lens = torch.from_numpy(wl.context_lens).to(cuda_device)
        qd = q.to(cuda_device)
        _status_clear()
        for rows in (slice(0, na), slice(0, wl.batch)):
            nb = rows.stop
            out = torch.full((nb, H, 128), float("nan"), device=cuda_device)
            B.pa_decode_attention_partitioned(out, qd[rows].contiguous(), gp.h, 0,
                                              tables[rows].contiguous(), wl.max_blocks,
                                              lens[rows].contiguous(), nb, 16, H, 1, 128,
                                              wl.scale, 0, ws, need)
            torch.cuda.synchronize()
            assert max_abs_err(out, ref[:nb]) <= TOL, nb
        assert B.pa_get_status() == 0
        out = torch.zeros((wl.batch, H, 128), device=cuda_device)
        with pytest.raises(B.PagedAttnError) as e:
            B.pa_decode_attention_partitioned(out, qd, gp.h, 0, tables, wl.max_blocks, lens,
                                              wl.batch, 16, H, 1, 128, wl.scale, 0, ws, need - 1)
        assert e.value.code == B.PA_ERR_WORKSPACE
    finally:
        gp.close()
