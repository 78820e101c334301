"""GPU parity for the layout variants (separate K/V caches, layer-major stacks)
and for the append fused into decode, against the oracle on the equivalent
fused pool."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W
from gpu_helpers import GpuPool, device_tables, gpu_decode, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu


def _split(fused, layout):
    """Separate K and V tensors holding the same rows as the fused pool
    [nb, 2, L, Hkv, B, D] (torch re-layout of the input, not the CUDA path)."""
    if layout == "separate_kv":           # vllmini-style k_cache / v_cache [nb, Hkv, B, D] per layer
        assert fused.shape[2] == 1
        return fused[:, 0, 0].contiguous(), fused[:, 1, 0].contiguous()
    if layout == "layer_major":           # [L, nb, Hkv, B, D]
        return (fused[:, 0].permute(1, 0, 2, 3, 4).contiguous(),
                fused[:, 1].permute(1, 0, 2, 3, 4).contiguous())
    raise ValueError(layout)


def _strides(wl, layout):
    tile = wl.block_size * wl.head_dim
    if layout == "separate_kv":
        return wl.num_kv_heads * tile, 0, tile
    return wl.num_kv_heads * tile, wl.num_blocks * wl.num_kv_heads * tile, tile


def _fused_from(kc, vc, wl, layout):
    if layout == "separate_kv":
        return torch.stack([kc, vc], dim=1).unsqueeze(2)
    return torch.stack([kc.permute(1, 0, 2, 3, 4), vc.permute(1, 0, 2, 3, 4)], dim=1)


@pytest.mark.parametrize("layout,dtype,L", [("separate_kv", "f32", 1), ("separate_kv", "bf16", 1),
                                            ("layer_major", "bf16", 3)])
def test_strided_layouts_decode_append_gather(cuda_device, layout, dtype, L):
    wl = W.custom("strided", dtype, L, 16, 4, 128, 16, [1, 15, 16, 17, 200, 511, 0], seed=41,
                  spare_blocks=6, interleave=True, steps=1)
    fused = W.make_pool(wl)
    kc, vc = (t.to(cuda_device) for t in _split(fused, layout))
    sb, sl, sh = _strides(wl, layout)
    h = B.pa_pool_create_strided(kc, vc, sb, sl, sh, wl.num_blocks, L, wl.num_kv_heads,
                                 wl.block_size, wl.head_dim, kc.dtype)
    try:
        qs = W.make_queries(wl, L)
        bt, ln = device_tables(wl, cuda_device)
        tol = 1e-5 if dtype == "f32" else 2e-3

        class Handle:
            pass

        gp = Handle()
        gp.wl, gp.h = wl, h
        for layer in range(L):
            for pb in (0, 2):
                out = gpu_decode(gp, qs[layer].to(cuda_device), layer, bt, ln, partition_blocks=pb)
                assert max_abs_err(out, oracle_decode(wl, fused, qs[layer], layer)) <= tol
        # append into the last layer, then compare every byte via the fused view
        k, v = W.make_new_tokens(wl, 1)
        tables = wl.block_tables.copy()
        for b, n in enumerate(wl.context_lens):
            if n % wl.block_size == 0:
                tables[b, n // wl.block_size] = wl.free_stack.pop()
        btn = torch.from_numpy(tables).to(cuda_device)
        pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
        B.pa_write_kv(h, L - 1, k[0].to(cuda_device), v[0].to(cuda_device), btn, wl.max_blocks,
                      pos, wl.batch)
        host = W.as_oracle_array(fused).copy()
        oracle.write_kv(host, L - 1, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                        wl.context_lens)
        torch.cuda.synchronize()
        assert np.array_equal(W.as_oracle_array(_fused_from(kc, vc, wl, layout).cpu()), host)
        # gather from the strided layout
        T = int(wl.context_lens.max()) + 1
        lens1 = wl.context_lens + 1
        kg = torch.empty((wl.batch, T, wl.num_kv_heads, wl.head_dim), dtype=kc.dtype,
                         device=cuda_device)
        vg = torch.empty_like(kg)
        mg = torch.empty((wl.batch, T), dtype=torch.uint8, device=cuda_device)
        B.pa_gather_kv(kg, vg, mg, h, L - 1, btn, wl.max_blocks,
                       torch.from_numpy(lens1).to(cuda_device), wl.batch, T)
        kr, vr, mr = oracle.gather_kv(host, L - 1, tables, lens1, T)
        torch.cuda.synchronize()
        assert np.array_equal(W.as_oracle_array(kg), kr)
        assert np.array_equal(W.as_oracle_array(vg), vr)
        assert np.array_equal(mg.cpu().numpy().astype(bool), mr)
        assert B.pa_get_status() == 0
    finally:
        B.pa_pool_destroy(h)


@pytest.mark.parametrize("dtype,D,Bs,G,pb,kind", [("bf16", 128, 16, 4, 0, "AUTO"),
                                                  ("bf16", 128, 32, 1, 2, "AUTO"),
                                                  ("bf16", 64, 16, 8, 1, "AUTO"),
                                                  ("bf16", 128, 32, 4, 3, "CUDA_CORES"),
                                                  ("f32", 64, 16, 2, 3, "AUTO")])
def test_fused_append_decode_matches_separate_calls(cuda_device, dtype, D, Bs, G, pb, kind):
    Hkv = 2
    lens = [0, 1, Bs - 1, Bs, 3 * Bs, 3 * Bs + 1, 7 * Bs + 3]   # positions of the new token
    wl = W.custom("fused", dtype, 2, Hkv * G, Hkv, D, Bs, lens, seed=D + G + Bs, steps=1,
                  spare_blocks=3)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    k, v = W.make_new_tokens(wl, 1)
    tables = wl.block_tables.copy()
    for b, n in enumerate(wl.context_lens):
        if n % wl.block_size == 0:
            tables[b, n // wl.block_size] = wl.free_stack.pop()
    gp = GpuPool(wl, pool.to(cuda_device))
    B.pa_pool_set_decode_kernel(gp.h, getattr(B, "PA_DECODE_" + kind))
    bt = torch.from_numpy(tables).to(cuda_device)
    pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
    lens1 = wl.context_lens + 1
    ln1 = torch.from_numpy(lens1).to(cuda_device)
    out = torch.full((wl.batch, wl.num_heads, D), float("nan"), device=cuda_device)
    need = B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, wl.max_blocks, pb)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
    B.pa_write_kv_and_decode(out, q.to(cuda_device), gp.h, 1, k[0].to(cuda_device),
                             v[0].to(cuda_device), pos, bt, wl.max_blocks, ln1, wl.batch,
                             wl.block_size, wl.num_heads, Hkv, D, wl.scale, pb, ws, need)
    host = W.as_oracle_array(pool).copy()
    oracle.write_kv(host, 1, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                    wl.context_lens)
    ref = oracle.decode_attention(W.as_oracle_array(q), host, 1, tables, lens1, wl.num_heads,
                                  wl.scale)
    torch.cuda.synchronize()
    assert max_abs_err(out, ref) <= (1e-5 if dtype == "f32" else 2e-3)
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    assert B.pa_get_status() == 0


@pytest.mark.parametrize("kind", ["AUTO", "CUDA_CORES"])
def test_fused_append_position_past_context(cuda_device, kind):
    """A position outside the decoded context is still stored (by partition 0)
    and does not change the decode -- on the tensor-core and CUDA-core kernels."""
    wl = W.custom("past", "bf16", 1, 8, 2, 128, 16, [40, 70], seed=3, spare_blocks=2)
    pool = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    k, v = W.make_new_tokens(wl, 1)
    gp = GpuPool(wl, pool.to(cuda_device))
    B.pa_pool_set_decode_kernel(gp.h, getattr(B, "PA_DECODE_" + kind))
    bt, ln = device_tables(wl, cuda_device)
    pos_h = np.array([45, 75], np.int32)                      # beyond n, inside the last block
    out = torch.empty((2, 8, 128), device=cuda_device)
    need = B.pa_decode_workspace_size(gp.h, 2, 8, wl.max_blocks, 1)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
    B.pa_write_kv_and_decode(out, q.to(cuda_device), gp.h, 0, k[0].to(cuda_device),
                             v[0].to(cuda_device), torch.from_numpy(pos_h).to(cuda_device), bt,
                             wl.max_blocks, ln, 2, 16, 8, 2, 128, wl.scale, 1, ws, need)
    host = W.as_oracle_array(pool).copy()
    ref = oracle.decode_attention(W.as_oracle_array(q), host, 0, wl.block_tables,
                                  wl.context_lens, 8, wl.scale)
    oracle.write_kv(host, 0, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), wl.block_tables,
                    pos_h)
    torch.cuda.synchronize()
    assert max_abs_err(out, ref) <= 2e-3
    assert np.array_equal(W.as_oracle_array(gp.t), host)
    assert B.pa_get_status() == 0
