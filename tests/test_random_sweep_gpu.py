"""Seeded randomized parity sweep on the GPU: random shapes (dtype, head_dim,
block size, GQA group 1-8, 16, 24, 32, 48, 64, KV heads, batch, ragged lengths with 0 / 1 /
block multiples), random layer, partition size, pool layout and decode kernel (CUDA cores,
mma.sync, tcgen05), plus the fused append path -- each case against the oracle on the same
inputs.  A second seeded set draws the large groups (96, 128, 192 query heads per KV head)
that the tcgen05 kernel serves as sibling chunk CTAs."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_239_gb300 import binding as B
from paged_kv_cache_239_gb300 import workloads as W
from gpu_helpers import TOL, max_abs_err, pool_in_layout

pytestmark = pytest.mark.gpu

N_CASES = 112
N_LARGE = 12


def _case(i):
    rng = np.random.default_rng(1000 + i)
    dtype = "f32" if rng.random() < 0.25 else "bf16"
    D = int(rng.choice([64, 128]))
    Bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8])) if dtype == "f32" else \
        int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 16, 24, 32, 48, 64]))
    L = int(rng.integers(1, 4))
    batch = int(rng.integers(1, 10))
    special = [0, 1, Bs - 1, Bs, Bs + 1, 2 * Bs]
    lens = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(0, 20 * Bs))
            for _ in range(batch)]
    layout = str(rng.choice(["fused", "separate", "layer_major"]))
    if layout == "separate":
        L = 1
    return rng, dtype, D, Bs, Hkv, G, L, lens, layout


def _large_case(i):
    rng = np.random.default_rng(5000 + i)
    Bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([96, 128, 192]))
    L = int(rng.integers(1, 3))
    batch = int(rng.integers(1, 8))
    special = [0, 1, Bs - 1, Bs, Bs + 1, 2 * Bs, 128, 129]
    lens = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(0, 40 * Bs))
            for _ in range(batch)]
    layout = str(rng.choice(["fused", "separate", "layer_major"]))
    if layout == "separate":
        L = 1
    return rng, "bf16", 128, Bs, Hkv, G, L, lens, layout


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(cuda_device, i):
    _run_case(cuda_device, i, *_case(i))


@pytest.mark.parametrize("i", range(N_LARGE))
def test_random_large_group_matches_oracle(cuda_device, i):
    _run_case(cuda_device, 1000 + i, *_large_case(i))


def _run_case(cuda_device, i, rng, dtype, D, Bs, Hkv, G, L, lens, layout):
    H = Hkv * G
    wl = W.custom(f"rnd{i}", dtype, L, H, Hkv, D, Bs, lens, seed=2000 + i,
                  spare_blocks=int(rng.integers(0, 5)), interleave=bool(rng.random() < 0.5),
                  steps=1)
    fused = W.make_pool(wl)
    q = W.make_queries(wl, 1)[0]
    keep, h = pool_in_layout(wl, fused, layout, cuda_device)
    try:
        kinds = [B.PA_DECODE_AUTO]
        if dtype == "bf16":
            kinds.append(B.PA_DECODE_CUDA_CORES)
        if dtype == "bf16":
            kinds.append(B.PA_DECODE_TENSOR_CORES)
        if dtype == "bf16" and D == 128 and G % 16 == 0:
            kinds.append(B.PA_DECODE_TCGEN05)
        layer = int(rng.integers(0, L))
        pb = int(rng.choice([0, 1, 2, 3, wl.max_blocks]))
        bt = torch.from_numpy(wl.block_tables).to(cuda_device)
        ln = torch.from_numpy(wl.context_lens).to(cuda_device)
        qd = q.to(cuda_device)
        ref = oracle.decode_attention(W.as_oracle_array(q), W.as_oracle_array(fused), layer,
                                      wl.block_tables, wl.context_lens, H, wl.scale)
        for kind in kinds:
            B.pa_pool_set_decode_kernel(h, kind)
            need = B.pa_decode_workspace_size(h, wl.batch, H, wl.max_blocks, pb)
            ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)
            out = torch.full((wl.batch, H, D), float("nan"), device=cuda_device)
            B.pa_decode_attention_partitioned(out, qd, h, layer, bt, wl.max_blocks, ln, wl.batch,
                                              Bs, H, Hkv, D, wl.scale, pb, ws, need)
            torch.cuda.synchronize()
            err = max_abs_err(out, ref)
            assert err <= TOL[dtype], (i, kind, dtype, D, Bs, Hkv, G, layout, pb, err)
        B.pa_pool_set_decode_kernel(h, B.PA_DECODE_AUTO)
        need = B.pa_decode_workspace_size(h, wl.batch, H, wl.max_blocks, pb)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda_device)

        # fused append at position n (a new block where n % B == 0), decode over n + 1
        k, v = W.make_new_tokens(wl, 1)
        tables = wl.block_tables.copy()
        for b, n in enumerate(wl.context_lens):
            if n % Bs == 0:
                tables[b, n // Bs] = wl.free_stack.pop()
        btn = torch.from_numpy(tables).to(cuda_device)
        pos = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
        lens1 = wl.context_lens + 1
        out = torch.full((wl.batch, H, D), float("nan"), device=cuda_device)
        B.pa_write_kv_and_decode(out, qd, h, layer, k[0].to(cuda_device), v[0].to(cuda_device),
                                 pos, btn, wl.max_blocks, torch.from_numpy(lens1).to(cuda_device),
                                 wl.batch, Bs, H, Hkv, D, wl.scale, pb, ws, need)
        host = W.as_oracle_array(fused).copy()
        oracle.write_kv(host, layer, W.as_oracle_array(k[0]), W.as_oracle_array(v[0]), tables,
                        wl.context_lens)
        ref1 = oracle.decode_attention(W.as_oracle_array(q), host, layer, tables, lens1, H,
                                       wl.scale)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref1) <= TOL[dtype], (i, "fused")
        assert B.pa_get_status() == 0
    finally:
        B.pa_pool_destroy(h)
