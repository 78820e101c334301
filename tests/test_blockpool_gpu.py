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


@pytest.mark.parametrize("kind", ["auto", "cuda_cores", "tensor_cores"])
def test_blockpool_device_loop_fused(cuda_device, kind):
    """The device free stack and the fused append + decode through BlockPool:
    every step allocates on the device, appends and decodes in one launch;
    tables, pool and outputs match the host allocator + oracle."""
    nb, Bs, Hkv, D, H, batch, steps = 48, 16, 2, 64, 16, 5, 37
    pool = BlockPool(num_blocks=nb, block_size=Bs, num_layers=1, num_kv_heads=Hkv, head_dim=D,
                     dtype=torch.bfloat16, device=cuda_device)
    pool.set_decode_kernel(kind)
    ref = FreeBlockStack(nb)
    stack = pool.device_stack()
    g = torch.Generator().manual_seed(11)
    tables = np.full((batch, 8), -1, np.int32)
    lens = np.zeros(batch, np.int32)
    bt = torch.from_numpy(tables.copy()).to(cuda_device)
    host = W.as_oracle_array(pool.pool.cpu()).copy()
    for step in range(steps):
        pos = torch.from_numpy(lens.copy()).to(cuda_device)
        pool.device_allocate_blocks(stack, bt, pos)
        for b in range(batch):
            if lens[b] % Bs == 0:
                tables[b, lens[b] // Bs] = ref.allocate_block()
        k = torch.randn(batch, Hkv, D, generator=g).bfloat16()
        v = torch.randn(batch, Hkv, D, generator=g).bfloat16()
        q = torch.randn(batch, H, D, generator=g).bfloat16()
        oracle.write_kv(host, 0, W.as_oracle_array(k), W.as_oracle_array(v), tables, lens)
        lens = lens + 1
        out = pool.write_kv_and_decode(q.to(cuda_device), 0, k.to(cuda_device), v.to(cuda_device),
                                       pos, bt, torch.from_numpy(lens).to(cuda_device),
                                       scale=D ** -0.5, partition_blocks=1)
        if step in (0, 15, 16, steps - 1):
            ref_out = oracle.decode_attention(W.as_oracle_array(q), host, 0, tables, lens, H,
                                              D ** -0.5)
            assert max_abs_err(out, ref_out) <= 2e-3, step
    torch.cuda.synchronize()
    assert np.array_equal(bt.cpu().numpy(), tables)
    assert np.array_equal(W.as_oracle_array(pool.pool.cpu()), host)
    # finish two sequences on the device; the stack comes back in the host's order
    finished = torch.tensor([1, 0, 0, 1, 0], dtype=torch.uint8, device=cuda_device)
    pool.device_free_blocks(stack, bt, torch.from_numpy(lens).to(cuda_device), finished)
    for b in (0, 3):
        for j in range(-(-int(lens[b]) // Bs)):
            ref.free_block(int(tables[b, j]))
            tables[b, j] = -1
    torch.cuda.synchronize()
    assert np.array_equal(bt.cpu().numpy(), tables)
    pool.download_device_stack(stack)
    assert pool.num_free() == ref.num_free()
    assert [pool.allocate_block() for _ in range(ref.num_free())] == \
        [ref.allocate_block() for _ in range(ref.num_free())]
    pool.close()
