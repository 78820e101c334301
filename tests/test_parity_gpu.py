"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Attention within 1e-5 (fp32 inputs) / 2e-3 (bf16 inputs,
fp32 accumulation) max-abs; append and gather bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.allocator import FreeBlockStack
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W
from gpu_helpers import (TOL, GpuPool, device_tables, gpu_decode, layer_subpool, max_abs_err,
                         oracle_decode)

pytestmark = pytest.mark.gpu


def _check_status(expected=0):
    st = B.pa_get_status()
    assert st == expected, f"device status {st:#x}, expected {expected:#x}"


# ---------------------------------------------------------------- small grid

GRID = []
for dtype in ("f32", "bf16"):
    for D in (64, 128):
        for Bs in (16, 32):
            for G in (1, 2, 4, 8):
                GRID.append((dtype, D, Bs, G))


@pytest.mark.parametrize("dtype,D,Bs,G", GRID)
def test_decode_grid_all_partitionings(cuda_device, dtype, D, Bs, G):
    Hkv = 2
    lens = [1, Bs - 1, Bs, Bs + 1, 3 * Bs + 5, 9 * Bs, 9 * Bs + 7, 0, 2]
    wl = W.custom("grid", dtype, 2, Hkv * G, Hkv, D, Bs, lens, seed=D + Bs + G, spare_blocks=5,
                  interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    qd = q.to(cuda_device)
    ref = oracle_decode(wl, pool, q, 1)
    kinds = [B.PA_DECODE_TENSOR_CORES, B.PA_DECODE_CUDA_CORES] if dtype == "bf16" else \
        [B.PA_DECODE_AUTO]
    for kind in kinds:
        B.pa_pool_set_decode_kernel(gp.h, kind)
        for pb in (0, 1, 2, 3, wl.max_blocks):
            out = gpu_decode(gp, qd, 1, bt, ln, partition_blocks=pb)
            torch.cuda.synchronize()
            err = max_abs_err(out, ref)
            assert err <= TOL[dtype], f"kernel {kind}, partition_blocks={pb}: max abs err {err}"
            assert torch.isfinite(out).all()
    if dtype == "f32":
        B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_TENSOR_CORES)
        with pytest.raises(B.PagedAttnError) as e:
            gpu_decode(gp, qd, 1, bt, ln)
        assert e.value.code == B.PA_ERR_UNSUPPORTED
    _check_status()
    gp.close()


def test_decode_tiny_f32_named(cuda_device):
    wl = W.named(1)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
    ref = oracle_decode(wl, pool, q, 0)
    assert max_abs_err(out, ref) <= 1e-5
    _check_status()


def test_decode_mini_infer_all_layers(cuda_device):
    wl = W.named(2)
    pool = W.make_pool(wl)
    qs = W.make_queries(wl, wl.num_layers)
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    qd = qs.to(cuda_device)
    worst = 0.0
    for layer in range(wl.num_layers):
        out = gpu_decode(gp, qd[layer], layer, bt, ln)
        ref = oracle_decode(wl, pool, qs[layer], layer)
        worst = max(worst, max_abs_err(out, ref))
    assert worst <= 2e-3, worst
    _check_status()


def test_decode_long_context_split(cuda_device):
    wl = W.named(4)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    pb = B.pa_decode_partition_blocks(gp.h, wl.batch, wl.num_heads, wl.max_blocks)
    assert pb < wl.max_blocks, "the long-context workload must take the split path"
    ref = oracle_decode(wl, pool, q, 0)
    for kind in (B.PA_DECODE_AUTO, B.PA_DECODE_CUDA_CORES):
        B.pa_pool_set_decode_kernel(gp.h, kind)
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
        assert max_abs_err(out, ref) <= 2e-3, kind
    _check_status()


@pytest.mark.slow
def test_decode_large_batch_every_sequence(cuda_device):
    """Full-size large-batch workload (about 71 GB of pool) in the launch
    configuration the benchmark times: every sequence and head of the first
    and the last layer against the oracle, element by element, on the
    automatic kernel and the CUDA-core kernel; then the benchmark's own call
    (the new token appended at the last context slot inside the decode
    launch) on the last layer, the whole layer's pool bytes compared too."""
    wl = W.named(3)
    pool = W.make_pool(wl, device=cuda_device)
    qs = W.make_queries(wl, 2, device=cuda_device)
    ks, vs = W.make_new_tokens(wl, 1, device=cuda_device)
    gp = GpuPool(wl, pool)
    bt, ln = device_tables(wl, cuda_device)
    last = wl.num_layers - 1
    for layer in (0, last):
        q = qs[layer % 2]
        sub, rows = layer_subpool(wl, pool, layer)
        ref = oracle.decode_attention(W.as_oracle_array(q.cpu()), W.as_oracle_array(sub), 0,
                                      rows, wl.context_lens, wl.num_heads, wl.scale)
        for kind in (B.PA_DECODE_AUTO, B.PA_DECODE_CUDA_CORES):
            B.pa_pool_set_decode_kernel(gp.h, kind)
            out = gpu_decode(gp, q, layer, bt, ln)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            err = max_abs_err(out, ref)
            assert err <= 2e-3, (layer, kind, err)
    _check_status()

    # the benchmark's step for one layer: append at position n - 1, decode over n
    B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_AUTO)
    sub, rows = layer_subpool(wl, pool, last)
    host = W.as_oracle_array(sub).copy()
    pos = (ln - 1).contiguous()
    oracle.write_kv(host, 0, W.as_oracle_array(ks[0].cpu()), W.as_oracle_array(vs[0].cpu()), rows,
                    wl.context_lens - 1)
    ref = oracle.decode_attention(W.as_oracle_array(qs[1].cpu()), host, 0, rows,
                                  wl.context_lens, wl.num_heads, wl.scale)
    need = B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, wl.max_blocks, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
    out = torch.full((wl.batch, wl.num_heads, wl.head_dim), float("nan"), device=cuda_device)
    B.pa_write_kv_and_decode(out, qs[1], gp.h, last, ks[0], vs[0], pos, bt, wl.max_blocks, ln,
                             wl.batch, wl.block_size, wl.num_heads, wl.num_kv_heads,
                             wl.head_dim, wl.scale, 0, ws, need)
    torch.cuda.synchronize()
    err = max_abs_err(out, ref)
    assert err <= 2e-3, err
    after, _ = layer_subpool(wl, pool, last)
    assert np.array_equal(W.as_oracle_array(after), host), "appended layer differs from the oracle"
    _check_status()
    gp.close()
    del pool
    torch.cuda.empty_cache()


def test_append_decode_loop(cuda_device):
    """Workload 5: per step, take a block on a boundary crossing (library
    allocator on GPU side, oracle free stack on CPU side), append one token,
    decode over n+1 tokens."""
    wl = W.named(5)
    pool = W.make_pool(wl)
    ks, vs = W.make_new_tokens(wl, wl.steps)
    qs = W.make_queries(wl, wl.steps)
    gp = GpuPool(wl, pool.to(cuda_device))
    host_pool = W.as_oracle_array(pool).copy()
    # both allocators start from the same free stack (ids still free, pop order)
    # (the stack's END is popped first: the in-use ids go last and are popped away)
    used = sorted(int(x) for x in wl.block_tables[wl.block_tables >= 0])
    full_order = list(wl.free_stack) + used
    B.pa_pool_seed_free_stack(gp.h, full_order)
    for _ in range(len(used)):
        B.pa_alloc_block(gp.h)
    ref_alloc = FreeBlockStack(wl.num_blocks)
    ref_alloc.seed(full_order)
    for _ in range(len(used)):
        ref_alloc.allocate_block()
    tables = wl.block_tables.copy()
    lens = wl.context_lens.copy()
    bt = torch.from_numpy(tables).to(cuda_device)
    kd, vd, qd = ks.to(cuda_device), vs.to(cuda_device), qs.to(cuda_device)
    check_steps = {0, 1, 30, 31, 32, 33, 63}
    for step in range(wl.steps):
        for b in range(wl.batch):
            if lens[b] % wl.block_size == 0:
                gid = B.pa_alloc_block(gp.h)
                assert gid == ref_alloc.allocate_block()
                tables[b, lens[b] // wl.block_size] = gid
        bt.copy_(torch.from_numpy(tables))
        pos = torch.from_numpy(lens.copy()).to(cuda_device)
        B.pa_write_kv(gp.h, 0, kd[step], vd[step], bt, wl.max_blocks, pos, wl.batch)
        oracle.write_kv(host_pool, 0, W.as_oracle_array(ks[step]), W.as_oracle_array(vs[step]),
                        tables, lens)
        lens = lens + 1
        ln = torch.from_numpy(lens.copy()).to(cuda_device)
        out = gpu_decode(gp, qd[step], 0, bt, ln)
        if step in check_steps:
            ref = oracle.decode_attention(W.as_oracle_array(qs[step]), host_pool, 0, tables, lens,
                                          wl.num_heads, wl.scale)
            assert max_abs_err(out, ref) <= 2e-3, step
    torch.cuda.synchronize()
    assert np.array_equal(W.as_oracle_array(gp.t), host_pool), "pool bytes differ after appends"
    _check_status()


# ---------------------------------------------------------------- append / gather


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_write_kv_bit_exact(cuda_device, cfg):
    wl = W.named(cfg)
    if cfg == 3:  # same geometry, small pool: the append does not depend on pool size
        wl = W.custom("wk3", "bf16", 32, 32, 8, 128, 16, wl.context_lens[:64], seed=5)
    pool = W.make_pool(wl)
    ks, vs = W.make_new_tokens(wl, 1)
    layer = wl.num_layers - 1
    # positions: the last cached slot of each sequence (always inside its table)
    pos = np.maximum(wl.context_lens - 1, 0).astype(np.int32)
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, _ = device_tables(wl, cuda_device)
    B.pa_write_kv(gp.h, layer, ks[0].to(cuda_device), vs[0].to(cuda_device), bt, wl.max_blocks,
                  torch.from_numpy(pos).to(cuda_device), wl.batch)
    host = W.as_oracle_array(pool).copy()
    oracle.write_kv(host, layer, W.as_oracle_array(ks[0]), W.as_oracle_array(vs[0]),
                    wl.block_tables, pos)
    torch.cuda.synchronize()
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    _check_status()


@pytest.mark.parametrize("cfg", [1, 2, 5])
def test_gather_kv_bit_exact(cuda_device, cfg):
    wl = W.named(cfg)
    pool = W.make_pool(wl)
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    T = int(wl.context_lens.max()) + 3
    layer = wl.num_layers // 2
    k_ref, v_ref, m_ref = oracle.gather_kv(W.as_oracle_array(pool), layer, wl.block_tables,
                                           wl.context_lens, T)
    dt = W.torch_dtype(wl)
    shape = (wl.batch, T, wl.num_kv_heads, wl.head_dim)
    k = torch.full(shape, 7, dtype=dt, device=cuda_device)
    v = torch.full(shape, 7, dtype=dt, device=cuda_device)
    m = torch.full((wl.batch, T), 9, dtype=torch.uint8, device=cuda_device)
    B.pa_gather_kv(k, v, m, gp.h, layer, bt, wl.max_blocks, ln, wl.batch, T)
    torch.cuda.synchronize()
    assert np.array_equal(W.as_oracle_array(k), k_ref)
    assert np.array_equal(W.as_oracle_array(v), v_ref)
    assert np.array_equal(m.cpu().numpy().astype(bool), m_ref)
    _check_status()


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token_is_exact(cuda_device, dtype):
    wl = W.custom("one", dtype, 1, 8, 2, 128, 16, [1, 1, 1, 1], seed=3, spare_blocks=3)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln).cpu()
    ref = oracle_decode(wl, pool, q, 0)
    assert np.array_equal(out.double().numpy(), ref)


def test_empty_and_full_tables(cuda_device):
    Bs, maxb = 16, 6
    lens = [0, maxb * Bs, 0, maxb * Bs - 1]
    wl = W.custom("edge", "bf16", 1, 8, 2, 64, Bs, lens, seed=12, max_blocks=maxb)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    ref = oracle_decode(wl, pool, q, 0)
    for pb in (0, 1, 4):
        out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb)
        o = out.cpu()
        assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
        assert max_abs_err(o, ref) <= 2e-3
    _check_status()


def test_zero_scale_and_batch_zero(cuda_device):
    wl = W.custom("z", "f32", 1, 4, 2, 64, 16, [5, 40], seed=2)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, scale=0.0)
    ref = oracle_decode(wl, pool, q, 0, scale=0.0)
    assert max_abs_err(out, ref) <= 1e-5
    # batch 0 launches nothing
    B.pa_decode_attention(None, None, gp.h, 0, None, 4, None, 0, 16, 4, 2, 64, 1.0, None, 0)
    _check_status()


def test_bad_block_id_is_flagged_not_faulted(cuda_device):
    wl = W.custom("bad", "bf16", 1, 4, 2, 64, 16, [40, 40, 40], seed=6, spare_blocks=2)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    tables = wl.block_tables.copy()
    tables[1, 1] = wl.num_blocks + 1000   # out of range
    tables[2, 2] = -5
    bt = torch.from_numpy(tables).to(cuda_device)
    ln = torch.from_numpy(wl.context_lens).to(cuda_device)
    _check_status()
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln).cpu()
    st = B.pa_get_status()
    assert st & B.PA_STATUS_BAD_BLOCK_ID
    ref = oracle_decode(wl, pool, q, 0)
    assert max_abs_err(out[0], ref[0]) <= 2e-3   # untouched sequence is still right
    assert torch.isfinite(out).all()
    # append through a bad id is skipped and flagged
    k, v = W.make_new_tokens(wl, 1)
    before = gp.t.clone()
    B.pa_write_kv(gp.h, 0, k[0].to(cuda_device), v[0].to(cuda_device), bt, wl.max_blocks,
                  torch.tensor([20, 20, 39], dtype=torch.int32, device=cuda_device), 3)
    st = B.pa_get_status()
    assert st & B.PA_STATUS_BAD_BLOCK_ID
    changed = (gp.t != before).reshape(wl.num_blocks, -1).any(dim=1).nonzero().flatten().tolist()
    assert changed == [int(tables[0, 1])]


def test_bad_length_is_flagged(cuda_device):
    wl = W.custom("len", "bf16", 1, 4, 2, 64, 16, [20, 20], seed=7)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, _ = device_tables(wl, cuda_device)
    ln = torch.tensor([20, wl.max_blocks * 16 + 1], dtype=torch.int32, device=cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln).cpu()
    assert B.pa_get_status() & B.PA_STATUS_BAD_LENGTH
    assert torch.all(out[1] == 0)


def _without_blocks(wl, tables, bad):
    """The tables with the blocks listed in bad[b] (logical indices) removed
    and the lengths shortened by their tokens: the attention the kernels give
    when those blocks' ids are out of range (their tokens get no weight)."""
    lens = wl.context_lens.copy()
    out = np.full_like(tables, -1)
    for b in range(wl.batch):
        n = int(lens[b])
        keep = [j for j in range(-(-n // wl.block_size)) if j not in bad.get(b, ())]
        lost = sum(min(wl.block_size, n - j * wl.block_size) for j in bad.get(b, ()))
        out[b, :len(keep)] = tables[b, keep]
        lens[b] = n - lost
    return out, lens


@pytest.mark.parametrize("H,Hkv", [(32, 1), (32, 8)])
def test_tokens_of_bad_blocks_get_no_weight(cuda_device, H, Hkv):
    """A table entry outside [0, num_blocks) is flagged, and every kernel gives
    its block's tokens no weight: the result is the attention over the other
    tokens (the oracle on the same tables with those blocks removed), and a
    sequence with no valid token left gives a zero vector.  The cases: the
    whole first 128-token tile of a context, one block inside it, two whole
    tiles and a ragged last block, and every block."""
    lens = [600, 300, 1000, 130]
    wl = W.custom("badw", "bf16", 1, H, Hkv, 128, 16, lens, seed=31, spare_blocks=4)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        tables = wl.block_tables.copy()
        bad = {0: tuple(range(8)), 1: (5,), 2: tuple(range(8, 24)) + (62,),
               3: tuple(range(-(-130 // 16)))}
        for b, js in bad.items():
            for k, j in enumerate(js):
                tables[b, j] = (-1 - k) if k % 2 else wl.num_blocks + 3 * k
        ref_tables, ref_lens = _without_blocks(wl, wl.block_tables, bad)
        assert ref_lens[3] == 0
        ref = oracle_decode(wl, pool, q, 0, tables=ref_tables, lens=ref_lens)
        bt = torch.from_numpy(tables).to(cuda_device)
        ln = torch.from_numpy(wl.context_lens).to(cuda_device)
        kinds = [B.PA_DECODE_AUTO, B.PA_DECODE_TENSOR_CORES, B.PA_DECODE_CUDA_CORES]
        if B.pa_decode_kernel_choice(gp.h, H) == B.PA_DECODE_TCGEN05:
            kinds.append(B.PA_DECODE_TCGEN05)
        torch.cuda.synchronize()
        B.pa_get_status()
        for kind in kinds:
            B.pa_pool_set_decode_kernel(gp.h, kind)
            for pb in (0, 1, 3, wl.max_blocks):
                out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb).cpu()
                assert B.pa_get_status() == B.PA_STATUS_BAD_BLOCK_ID, (kind, pb)
                assert torch.isfinite(out).all(), (kind, pb)
                assert max_abs_err(out, ref) <= TOL["bf16"], (kind, pb)
                assert torch.all(out[3] == 0), (kind, pb)
    finally:
        gp.close()


def test_decode_on_side_stream_matches(cuda_device):
    wl = W.custom("stream", "bf16", 2, 16, 4, 128, 32, [100, 250, 3, 64], seed=13)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    s = torch.cuda.Stream()
    qd = q.to(cuda_device)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = gpu_decode(gp, qd, 1, bt, ln, stream=s, partition_blocks=2)
    s.synchronize()
    assert max_abs_err(out, oracle_decode(wl, pool, q, 1)) <= 2e-3
    _check_status()


def test_append_and_decode_captured_in_cuda_graph(cuda_device):
    """One step (append + decode for every layer) captured into a CUDA graph
    and replayed: same results as the oracle, status clean."""
    wl = W.custom("graph", "bf16", 3, 16, 4, 128, 16, [40, 300, 17, 1000], seed=31, steps=1)
    pool = W.make_pool(wl)
    qs = W.make_queries(wl, 3)
    ks, vs = W.make_new_tokens(wl, 3)
    gp = GpuPool(wl, pool.to(cuda_device))
    tables = wl.block_tables.copy()
    for b, n in enumerate(wl.context_lens):
        if n % wl.block_size == 0:
            tables[b, n // wl.block_size] = wl.free_stack.pop()
    bt = torch.from_numpy(tables).to(cuda_device)
    pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
    lens1 = torch.from_numpy(wl.context_lens + 1).to(cuda_device)
    qd, kd, vd = qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device)
    outs = torch.zeros((3, wl.batch, wl.num_heads, wl.head_dim), dtype=torch.float32,
                       device=cuda_device)
    pb = 4
    need = B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, wl.max_blocks, pb)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    B.pa_get_status()  # first launching-side call before capture (status word lookup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for l in range(3):
                B.pa_write_kv(gp.h, l, kd[l], vd[l], bt, wl.max_blocks, pos, wl.batch, stream=s)
                B.pa_decode_attention_partitioned(outs[l], qd[l], gp.h, l, bt, wl.max_blocks,
                                                  lens1, wl.batch, wl.block_size, wl.num_heads,
                                                  wl.num_kv_heads, wl.head_dim, wl.scale, pb,
                                                  ws, need, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.all(outs == 0), "capture must not execute the kernels"
    g.replay()
    g.replay()   # replaying twice rewrites the same slots: same result
    torch.cuda.synchronize()
    host = W.as_oracle_array(pool).copy()
    for l in range(3):
        oracle.write_kv(host, l, W.as_oracle_array(ks[l]), W.as_oracle_array(vs[l]), tables,
                        wl.context_lens)
    for l in range(3):
        ref = oracle.decode_attention(W.as_oracle_array(qs[l]), host, l, tables,
                                      wl.context_lens + 1, wl.num_heads, wl.scale)
        assert max_abs_err(outs[l], ref) <= 2e-3, l
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    _check_status()


def test_bounded_wait_times_out_into_status(cuda_device):
    """A barrier nothing completes: the bounded wait gives up, the status word
    says PA_STATUS_TIMEOUT, and a following decode still works."""
    assert B.pa_get_status() == 0
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    B.pa_selftest_wait_timeout()
    t1.record()
    assert B.pa_get_status() == B.PA_STATUS_TIMEOUT
    assert 10.0 <= t0.elapsed_time(t1) < 2000.0     # about the 20 ms limit
    assert B.pa_get_status() == 0                    # read-and-clear
    wl = W.custom("after", "bf16", 1, 8, 2, 128, 16, [30, 100], seed=2)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln)
    assert max_abs_err(out, oracle_decode(wl, pool, q, 0)) <= 2e-3
    _check_status()


@pytest.mark.parametrize("D,Bs", [(128, 16), (64, 32)])
def test_group_of_16_on_tensor_cores(cuda_device, D, Bs):
    """128 query heads over 8 KV heads style grouping (G = 16): two 8-head mma
    tiles per KV head; the CUDA-core kernel serves it as two 8-head chunks."""
    wl = W.custom("g16", "bf16", 2, 32, 2, D, Bs, [1, Bs, 5 * Bs + 3, 700, 0], seed=16,
                  spare_blocks=3, interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    ref = oracle_decode(wl, pool, q, 1)
    for pb in (0, 1, 3, wl.max_blocks):
        out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln, partition_blocks=pb)
        assert max_abs_err(out, ref) <= 2e-3, pb
    B.pa_pool_set_decode_kernel(gp.h, B.PA_DECODE_CUDA_CORES)
    for pb in (0, 1, wl.max_blocks):
        out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln, partition_blocks=pb)
        assert max_abs_err(out, ref) <= 2e-3, pb
    _check_status()


@pytest.mark.parametrize("Hkv,H,D,Bs", [(1, 24, 128, 16), (2, 64, 128, 32), (1, 32, 64, 16),
                                         (1, 64, 128, 16)])
def test_large_groups_in_head_chunks(cuda_device, Hkv, H, D, Bs):
    """Groups above 16 (multiples of 8, e.g. MQA with one KV head) run as 8- or
    16-head chunks of CTAs; every head matches the oracle, split or not, and
    the fused append works per chunked group."""
    wl = W.custom("bigg", "bf16", 2, H, Hkv, D, Bs, [1, Bs - 1, 3 * Bs, 9 * Bs + 5, 0, 400],
                  seed=H + D, spare_blocks=2, interleave=True, steps=1)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    ref = oracle_decode(wl, pool, q, 1)
    for pb in (0, 1, 4, wl.max_blocks):
        out = gpu_decode(gp, q.to(cuda_device), 1, bt, ln, partition_blocks=pb)
        assert max_abs_err(out, ref) <= 2e-3, pb
    k, v = W.make_new_tokens(wl, 1)
    tables = wl.block_tables.copy()
    for b, n in enumerate(wl.context_lens):
        if n % Bs == 0:
            tables[b, n // Bs] = wl.free_stack.pop()
    btn = torch.from_numpy(tables).to(cuda_device)
    pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
    lens1 = wl.context_lens + 1
    out = torch.full((wl.batch, H, D), float("nan"), device=cuda_device)
    need = B.pa_decode_workspace_size(gp.h, wl.batch, H, wl.max_blocks, 2)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
    B.pa_write_kv_and_decode(out, q.to(cuda_device), gp.h, 0, k[0].to(cuda_device),
                             v[0].to(cuda_device), pos, btn, wl.max_blocks,
                             torch.from_numpy(lens1).to(cuda_device), wl.batch, Bs, H, Hkv, D,
                             wl.scale, 2, ws, need)
    host = W.as_oracle_array(pool).copy()
    oracle.write_kv(host, 0, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                    wl.context_lens)
    ref1 = oracle.decode_attention(W.as_oracle_array(q), host, 0, tables, lens1, H, wl.scale)
    torch.cuda.synchronize()
    assert max_abs_err(out, ref1) <= 2e-3
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    _check_status()


@pytest.mark.parametrize("H,Hkv,D,Bs", [(71, 1, 128, 16), (232, 8, 128, 16), (12, 2, 64, 32),
                                        (20, 1, 64, 16), (11, 1, 128, 32)])
def test_groups_of_any_size_match_oracle(cuda_device, H, Hkv, D, Bs):
    """Groups that are no multiple of 8 (e.g. 71 query heads on one KV head, or
    232 on eight: 29 per group) run on the mma.sync kernel as 8-head chunks
    whose last holds the rest; every head, and no head of the next group, is
    written ("vllmini", "The CUDA Block Kernel": any num_heads over
    num_kv_heads).  Lengths around the blocks, every partitioning, the fused
    append's kernel and the wide CTAs (a whole table)."""
    lens = [0, 1, Bs - 1, Bs, Bs + 1, 5 * Bs + 3, 300, 40]
    wl = W.custom("anyg", "bf16", 1, H, Hkv, D, Bs, lens, seed=H * 7 + D + Bs, spare_blocks=3,
                  interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        assert B.pa_decode_kernel_choice(gp.h, H) == B.PA_DECODE_TENSOR_CORES
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        for kind in (B.PA_DECODE_AUTO, B.PA_DECODE_CUDA_CORES):
            B.pa_pool_set_decode_kernel(gp.h, kind)
            for pb in (0, 1, 2, wl.max_blocks):
                out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb)
                torch.cuda.synchronize()
                assert torch.isfinite(out).all(), (kind, pb)
                assert max_abs_err(out, ref) <= TOL["bf16"], (kind, pb)
        _check_status()
    finally:
        gp.close()


@pytest.mark.parametrize("H,Hkv,D,Bs", [(6, 2, 64, 16), (10, 2, 128, 32), (24, 2, 64, 16),
                                        (3, 1, 128, 16)])
def test_fp32_pools_any_group_match_oracle(cuda_device, H, Hkv, D, Bs):
    """fp32 pools run on the CUDA-core kernel, which serves any group in
    power-of-two head chunks (3 heads in a 4-head chunk, 5 in an 8-head one,
    12 as 8 + 4 of two 8-head chunks), the heads past the group masked; within
    the fp32 tolerance of the oracle at every partitioning."""
    lens = [0, 1, Bs - 1, Bs, Bs + 1, 4 * Bs + 5, 230]
    wl = W.custom("f32g", "f32", 1, H, Hkv, D, Bs, lens, seed=H * 11 + D, spare_blocks=2,
                  interleave=True)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    gp = GpuPool(wl, pool.to(cuda_device))
    try:
        assert B.pa_decode_kernel_choice(gp.h, H) == B.PA_DECODE_CUDA_CORES
        bt, ln = device_tables(wl, cuda_device)
        ref = oracle_decode(wl, pool, q, 0)
        for pb in (0, 1, 3, wl.max_blocks):
            out = gpu_decode(gp, q.to(cuda_device), 0, bt, ln, partition_blocks=pb)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all(), pb
            assert max_abs_err(out, ref) <= TOL["f32"], pb
        _check_status()
    finally:
        gp.close()
