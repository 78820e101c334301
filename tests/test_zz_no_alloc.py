"""pa_decode_attention_noalloc: decode for callers that cannot allocate device
memory while they run (an operator inside another engine that owns all device
memory and forbids cudaMalloc during its execution step).  Its split-K partials
live in a fixed device array compiled into the library instead of a caller's
workspace.  The source pages have no counterpart to this call.

The tests compare it, through the C ABI, with pa_decode_attention_partitioned
given an ordinary workspace, on two calls in a row (the second call must not be
disturbed by what the first left in the shared array); run a sequence of
differently cut calls against the one array -- the largest user of scratch
first, then shorter contexts, a tcgen05 call whose partials, descriptors and
cut records sit at other offsets, a call in wide CTAs that needs no scratch,
and an mma.sync call after them -- each against the fp64 oracle; and check
that calls needing more than the fixed array are refused before anything is
launched, with advice that fits the kernel.
This file is named to be collected last."""
import numpy as np
import pytest
import torch

from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W
from gpu_helpers import TOL, GpuPool, device_tables, gpu_decode, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc(gp, q, layer, bt, ln, partition_blocks):
    wl = gp.wl
    batch, H, D = q.shape
    out = torch.full((batch, H, D), float("nan"), dtype=torch.float32, device=q.device)
    B.pa_decode_attention_noalloc(out, q, gp.h, layer, bt, bt.shape[1], ln, batch,
                                  wl.block_size, H, wl.num_kv_heads, D, wl.scale,
                                  partition_blocks)
    return out


@pytest.mark.parametrize("partition_blocks,H,Hkv", [(3, 32, 8), (0, 32, 8),
                                                    (0, 64, 1), (0, 32, 2)])  # last two: tcgen05
def test_noalloc_matches_workspace_entry_point(cuda_device, partition_blocks, H, Hkv):
    wl = W.custom("noalloc", "bf16", 2, H, Hkv, 128, 32, [4000, 9000, 1, 700, 0, 2048, 33],
                  seed=77, spare_blocks=9)
    pool = W.make_pool(wl)
    qs = W.make_queries(wl, 2)
    gp = GpuPool(wl, pool.to(cuda_device))
    bt, ln = device_tables(wl, cuda_device)
    qd = qs.to(cuda_device)
    need = B.pa_decode_workspace_size(gp.h, wl.batch, wl.num_heads, wl.max_blocks,
                                      partition_blocks)
    assert 0 < need <= B.PA_NOALLOC_SCRATCH_BYTES, "the case must use split-K scratch"
    # two calls in a row: different layer and query, the array is reused
    for layer in (0, 1):
        ref = gpu_decode(gp, qd[layer], layer, bt, ln, partition_blocks=partition_blocks)
        got = _noalloc(gp, qd[layer], layer, bt, ln, partition_blocks)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert max_abs_err(got, ref.cpu().double().numpy()) <= TOL["bf16"], layer
    assert B.pa_get_status() == 0
    gp.close()


def test_noalloc_refuses_oversized_scratch(cuda_device):
    wl = W.custom("big", "bf16", 1, 32, 8, 128, 32, [131072] * 4, seed=5)
    pool = torch.zeros((1, 2, 1, 8, 32, 128), dtype=torch.bfloat16, device=cuda_device)
    h = B.pa_pool_create(pool, 1, 1, 8, 32, 128, pool.dtype)
    try:
        bt = torch.zeros((4, wl.max_blocks), dtype=torch.int32, device=cuda_device)
        ln = torch.zeros(4, dtype=torch.int32, device=cuda_device)
        out = torch.zeros((4, 32, 128), dtype=torch.float32, device=cuda_device)
        q = torch.zeros((4, 32, 128), dtype=torch.bfloat16, device=cuda_device)
        need = B.pa_decode_workspace_size(h, 4, 32, wl.max_blocks, 1)
        assert need > B.PA_NOALLOC_SCRATCH_BYTES
        with pytest.raises(B.PagedAttnError) as e:
            B.pa_decode_attention_noalloc(out, q, h, 0, bt, wl.max_blocks, ln, 4, 32, 32, 8,
                                          128, 1.0, 1)
        assert e.value.code == B.PA_ERR_WORKSPACE
        assert "scratch" in str(e.value)
        torch.cuda.synchronize()
        assert bool((out == 0).all())
    finally:
        B.pa_pool_destroy(h)


def test_noalloc_sequence_of_differently_cut_calls(cuda_device):
    """Calls of different shapes share the one array; each must read only what
    it wrote itself.  Order: most scratch first, so later calls run on top of
    larger leftovers."""
    steps = [  # (H, Hkv, lens, partition_blocks)
        (32, 8, [30000, 26000, 5000, 1], 1),        # mma.sync, one block per partition
        (32, 8, [3000, 1, 0, 300, 129], 0),          # mma.sync, heuristic partitions
        (64, 1, [4000, 9000, 1, 700, 0, 2048], 0),   # tcgen05, cut at CTA shares
        # wide mma.sync CTAs (8 x 8 KV heads: a third of a wave or more, tables
        # of 48 blocks): whole contexts, no scratch at all
        (16, 8, [1536, 1, 0, 700, 33, 1200, 64, 1535], 0),
        (32, 8, [4000, 2, 1500], 2),                 # mma.sync again, after tcgen05
    ]
    sizes = []
    for i, (H, Hkv, lens, pb) in enumerate(steps):
        wl = W.custom(f"seq{i}", "bf16", 1, H, Hkv, 128, 32, lens, seed=90 + i, spare_blocks=3,
                      interleave=True)
        pool = W.make_pool(wl)
        q = W.make_queries(wl, 1)[0]
        gp = GpuPool(wl, pool.to(cuda_device))
        bt, ln = device_tables(wl, cuda_device)
        need = B.pa_decode_workspace_size(gp.h, wl.batch, H, wl.max_blocks, pb)
        wide = H == 16
        if wide:   # (sequence, KV head) CTAs: between a third of the SMs and all of them
            sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
            assert sms <= wl.batch * Hkv * 3 and wl.batch * Hkv <= sms, sms
            assert B.pa_decode_partition_blocks(gp.h, wl.batch, H, wl.max_blocks) == wl.max_blocks
        assert (need == 0) if wide else (0 < need <= B.PA_NOALLOC_SCRATCH_BYTES), (i, need)
        sizes.append(need)
        got = _noalloc(gp, q.to(cuda_device), 0, bt, ln, pb)
        torch.cuda.synchronize()
        ref = oracle_decode(wl, pool, q, 0)
        assert torch.isfinite(got).all(), i
        assert max_abs_err(got, ref) <= TOL["bf16"], i
        assert B.pa_get_status() == 0
        gp.close()
    assert sizes[0] == max(sizes), sizes


def test_noalloc_refusal_advice_fits_the_kernel(cuda_device):
    """A tcgen05 call whose scratch exceeds the array is refused without the
    partition_blocks advice (that kernel ignores it); an mma.sync call keeps it.
    Refused calls launch nothing, so their device pointers are never read."""
    pool = torch.zeros((1, 2, 1, 1, 16, 128), dtype=torch.bfloat16, device=cuda_device)
    h = B.pa_pool_create(pool, 1, 1, 1, 16, 128, pool.dtype)
    try:
        batch = 4_000_000  # (sequence, head group) descriptors alone exceed 64 MiB
        assert B.pa_decode_kernel_choice(h, 64) == B.PA_DECODE_TCGEN05
        need = B.pa_decode_workspace_size(h, batch, 64, 1, 0)
        assert need > B.PA_NOALLOC_SCRATCH_BYTES
        lib = B.lib()
        fake = 0x7F0000000000
        rc = lib.pa_decode_attention_noalloc(fake, fake, h, 0, fake, 1, fake, batch, 16, 64, 1,
                                             128, 1.0, 0, None)
        assert rc == B.PA_ERR_WORKSPACE
        msg = B.last_error()
        assert "tcgen05" in msg and "caller-provided workspace" in msg
        assert "larger partition_blocks" not in msg
        B.pa_pool_set_decode_kernel(h, B.PA_DECODE_TENSOR_CORES)
        need = B.pa_decode_workspace_size(h, 64, 64, 1 << 14, 1)
        assert need > B.PA_NOALLOC_SCRATCH_BYTES
        rc = lib.pa_decode_attention_noalloc(fake, fake, h, 0, fake, 1 << 14, fake, 64, 16, 64,
                                             1, 128, 1.0, 1, None)
        assert rc == B.PA_ERR_WORKSPACE
        assert "larger partition_blocks" in B.last_error()
        torch.cuda.synchronize()
        assert B.pa_get_status() == 0
    finally:
        B.pa_pool_destroy(h)
