"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs."""
import math

import numpy as np
import torch

import oracle
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W

TOL = {"f32": 1e-5, "bf16": 2e-3}


class GpuPool:
    """A pool tensor on the GPU wrapped by a library handle."""

    def __init__(self, wl, pool_t):
        self.wl = wl
        self.t = pool_t
        self.h = B.pa_pool_create(pool_t, wl.num_blocks, wl.num_layers, wl.num_kv_heads,
                                  wl.block_size, wl.head_dim, pool_t.dtype)

    def close(self):
        if self.h:
            B.pa_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()


def pool_in_layout(wl, fused, layout, dev):
    """Device tensors holding the fused pool's rows in `layout` -- "fused"
    [n, 2, L, Hkv, B, D], "separate" K and V caches [n, Hkv, B, D] (one layer),
    "layer_major" K and V caches [L, n, Hkv, B, D] -- and a handle over them."""
    tile = wl.block_size * wl.head_dim
    if layout == "fused":
        t = fused.to(dev)
        return (t,), B.pa_pool_create(t, wl.num_blocks, wl.num_layers, wl.num_kv_heads,
                                      wl.block_size, wl.head_dim, t.dtype)
    if layout == "separate":
        kc, vc = fused[:, 0, 0].contiguous().to(dev), fused[:, 1, 0].contiguous().to(dev)
        sb, sl = wl.num_kv_heads * tile, 0
    else:
        kc = fused[:, 0].permute(1, 0, 2, 3, 4).contiguous().to(dev)
        vc = fused[:, 1].permute(1, 0, 2, 3, 4).contiguous().to(dev)
        sb, sl = wl.num_kv_heads * tile, wl.num_blocks * wl.num_kv_heads * tile
    h = B.pa_pool_create_strided(kc, vc, sb, sl, tile, wl.num_blocks, wl.num_layers,
                                 wl.num_kv_heads, wl.block_size, wl.head_dim, kc.dtype)
    return (kc, vc), h


def device_tables(wl, device):
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(device)
    lens = torch.from_numpy(np.ascontiguousarray(wl.context_lens)).to(device)
    return bt, lens


def gpu_decode(gp, q, layer, bt, lens, scale=None, partition_blocks=0, stream=None, out=None):
    wl = gp.wl
    batch, H, D = q.shape
    if out is None:
        out = torch.full((batch, H, D), float("nan"), dtype=torch.float32, device=q.device)
    need = B.pa_decode_workspace_size(gp.h, batch, H, bt.shape[1], partition_blocks)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device) if need else None
    B.pa_decode_attention_partitioned(out, q, gp.h, layer, bt, bt.shape[1], lens, batch,
                                      wl.block_size, H, wl.num_kv_heads, D,
                                      wl.scale if scale is None else scale, partition_blocks,
                                      ws, need, stream)
    return out


def oracle_decode(wl, pool_t, q_t, layer, tables=None, lens=None, scale=None):
    return oracle.decode_attention(W.as_oracle_array(q_t), W.as_oracle_array(pool_t), layer,
                                   wl.block_tables if tables is None else tables,
                                   wl.context_lens if lens is None else lens, wl.num_heads,
                                   wl.scale if scale is None else scale)


def layer_subpool(wl, pool_gpu, layer, tables=None, lens=None):
    """One layer of the blocks every sequence uses, copied to the host as a
    pool [n, 2, 1, Hkv, B, D] (the layer is sliced before the rows are picked,
    so a 71 GB pool costs one layer's bytes), with the tables renumbered to it:
    sequence b's blocks sit at consecutive ids in table order."""
    tables = wl.block_tables if tables is None else tables
    lens = wl.context_lens if lens is None else lens
    ids, rows = [], np.full(tables.shape, -1, np.int32)
    for b in range(len(lens)):
        nblk = -(-int(lens[b]) // wl.block_size)
        rows[b, :nblk] = np.arange(len(ids), len(ids) + nblk, dtype=np.int32)
        ids.extend(int(x) for x in tables[b, :nblk])
    idx = torch.tensor(ids, dtype=torch.long, device=pool_gpu.device)
    sub = pool_gpu[:, :, layer].index_select(0, idx).unsqueeze(2).contiguous().cpu()
    return sub, rows


def max_abs_err(gpu_out, ref):
    g = gpu_out.detach().cpu().double().numpy() if torch.is_tensor(gpu_out) else gpu_out
    return float(np.max(np.abs(g - ref))) if g.size else 0.0
