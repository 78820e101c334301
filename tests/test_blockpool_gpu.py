"""The BlockPool wrapper (mini-infer interface on the C ABI) end to end on
the GPU: allocate, append, decode, gather, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle.allocator import FreeBlockStack
from paged_kv_cache_239_gb300 import workloads as W
from paged_kv_cache_239_gb300.pool import BlockPool
from gpu_helpers import max_abs_err

pytestmark = pytest.mark.gpu


def test_blockpool_grow_append_decode_gather(cuda_device):
    nb, Bs, L, Hkv, D, H = 40, 16, 2, 2, 64, 16
    pool = BlockPool(num_blocks=nb, block_size=Bs, num_layers=L, num_kv_heads=Hkv, head_dim=D,
                     dtype=torch.bfloat16, device=cuda_device)
    ref = FreeBlockStack(nb)
    assert pool.block_bytes() == 2 * L * Hkv * Bs * D * 2
    batch, steps = 3, 40
    g = torch.Generator().manual_seed(3)
    tables = np.full((batch, 8), -1, np.int32)
    lens = np.zeros(batch, np.int32)
    host = W.as_oracle_array(pool.pool.cpu()).copy()     # zero-initialised like the page's pool
    assert not host.any()
    for step in range(steps):
        for b in range(batch):
            if lens[b] % Bs == 0:
                blk = pool.allocate_block()
                assert blk == ref.allocate_block()
                tables[b, lens[b] // Bs] = blk
        bt = torch.from_numpy(tables).to(cuda_device)
        pos = torch.from_numpy(lens.copy()).to(cuda_device)
        for layer in range(L):
            k = torch.randn(batch, Hkv, D, generator=g).bfloat16()
            v = torch.randn(batch, Hkv, D, generator=g).bfloat16()
            pool.write_kv(layer, k.to(cuda_device), v.to(cuda_device), bt, pos)
            oracle.write_kv(host, layer, W.as_oracle_array(k), W.as_oracle_array(v), tables, lens)
        lens = lens + 1
    ln = torch.from_numpy(lens).to(cuda_device)
    bt = torch.from_numpy(tables).to(cuda_device)
    q = torch.randn(batch, H, D, generator=g).bfloat16()
    for layer in range(L):
        out = pool.decode_attention(q.to(cuda_device), layer, bt, ln, scale=D ** -0.5)
        ref_out = oracle.decode_attention(W.as_oracle_array(q), host, layer, tables, lens, H,
                                          D ** -0.5)
        assert max_abs_err(out, ref_out) <= 2e-3
        out2 = pool.decode_attention(q.to(cuda_device), layer, bt, ln, scale=D ** -0.5,
                                     partition_blocks=1)
        assert max_abs_err(out2, ref_out) <= 2e-3
    kg, vg, mg = pool.gather_kv(1, bt, ln, 48)
    kr, vr, mr = oracle.gather_kv(host, 1, tables, lens, 48)
    assert np.array_equal(W.as_oracle_array(kg), kr) and np.array_equal(W.as_oracle_array(vg), vr)
    assert np.array_equal(mg.cpu().numpy(), mr)
    # finish sequence 1: its blocks go back on the stack, newest-freed first out
    for j in range(-(-int(lens[1]) // Bs)):
        pool.free_block(int(tables[1, j]))
        ref.free_block(int(tables[1, j]))
    assert pool.num_free() == ref.num_free()
    assert pool.allocate_block() == ref.allocate_block()
    assert np.array_equal(W.as_oracle_array(pool.pool), host)
    pool.close()
