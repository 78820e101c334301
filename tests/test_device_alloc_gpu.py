"""The free-block stack on the device against the oracle's free stack: batch
allocation / freeing must hand out and take back exactly the ids the same
sequence of host calls would (bit-exact tables and stack)."""
import numpy as np
import pytest
import torch

from oracle.allocator import FreeBlockStack
from paged_kv_cache_239_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _pool(dev, nb, Bs=16):
    t = torch.zeros((nb, 2, 1, 1, Bs, 64), dtype=torch.bfloat16, device=dev)
    return t, B.pa_pool_create(t, nb, 1, 1, Bs, 64, t.dtype)


class _null:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


def _download_stack(h, stack):
    B.pa_device_stack_download(h, stack)
    order = []
    while True:
        try:
            order.append(B.pa_alloc_block(h))
        except MemoryError:
            break
    return order   # pop order (top first)


@pytest.mark.parametrize("batch", [7, 1024, 3000])
def test_device_alloc_matches_host_pops(cuda_device, batch):
    Bs, maxb = 16, 8
    nb = batch * 3 + 5
    rng = np.random.default_rng(batch)
    pool_t, h = _pool(cuda_device, nb, Bs)
    ref = FreeBlockStack(nb)
    order = [int(x) for x in rng.permutation(nb)]
    try:
        B.pa_pool_seed_free_stack(h, order)
        ref.seed(order)
        stack = torch.empty(B.pa_device_stack_bytes(h) // 4, dtype=torch.int32, device=cuda_device)
        B.pa_device_stack_upload(h, stack)
        tables = np.full((batch, maxb), -1, np.int32)
        bt = torch.from_numpy(tables).to(cuda_device)
        for step in range(3):
            pos = rng.integers(0, maxb * Bs, size=batch).astype(np.int32)
            pos[:: 3] = (pos[:: 3] // Bs) * Bs           # a third start a new block
            B.pa_device_alloc_blocks(h, stack, bt, maxb, torch.from_numpy(pos).to(cuda_device),
                                     batch)
            for b in range(batch):
                if pos[b] % Bs == 0:
                    tables[b, pos[b] // Bs] = ref.allocate_block()
            torch.cuda.synchronize()
            assert np.array_equal(bt.cpu().numpy(), tables), step
        assert B.pa_get_status() == 0
        assert _download_stack(h, stack) == [ref.allocate_block() for _ in range(ref.num_free())]
    finally:
        B.pa_pool_destroy(h)


def test_device_alloc_exhaustion_flags_and_fills_minus_one(cuda_device):
    Bs, maxb, nb = 16, 4, 5
    pool_t, h = _pool(cuda_device, nb, Bs)
    try:
        stack = torch.empty(nb + 1, dtype=torch.int32, device=cuda_device)
        B.pa_device_stack_upload(h, stack)
        with pytest.raises(B.PagedAttnError):
            B.pa_alloc_block(h)                      # host allocator refused while lent
        pos = torch.zeros(8, dtype=torch.int32, device=cuda_device)
        bt = torch.full((8, maxb), -7, dtype=torch.int32, device=cuda_device)
        B.pa_device_alloc_blocks(h, stack, bt, maxb, pos, 8)
        got = bt[:, 0].cpu().tolist()
        assert got == [4, 3, 2, 1, 0, -1, -1, -1]
        assert B.pa_get_status() == B.PA_STATUS_NO_FREE_BLOCKS
        assert _download_stack(h, stack) == []
    finally:
        B.pa_pool_destroy(h)


def test_device_free_matches_host_frees(cuda_device):
    Bs, maxb, batch = 16, 6, 40
    nb = batch * maxb
    rng = np.random.default_rng(5)
    pool_t, h = _pool(cuda_device, nb, Bs)
    ref = FreeBlockStack(nb)
    try:
        lens = rng.integers(0, maxb * Bs + 1, size=batch).astype(np.int32)
        tables = np.full((batch, maxb), -1, np.int32)
        for b in range(batch):                       # host allocation for the initial tables
            for j in range(-(-int(lens[b]) // Bs)):
                tables[b, j] = B.pa_alloc_block(h)
                assert tables[b, j] == ref.allocate_block()
        finished = (rng.random(batch) < 0.4).astype(np.uint8)
        stack = torch.empty(nb + 1, dtype=torch.int32, device=cuda_device)
        B.pa_device_stack_upload(h, stack)
        bt = torch.from_numpy(tables).to(cuda_device)
        B.pa_device_free_blocks(h, stack, bt, maxb, torch.from_numpy(lens).to(cuda_device),
                                torch.from_numpy(finished).to(cuda_device), batch)
        for b in range(batch):
            if finished[b]:
                for j in range(-(-int(lens[b]) // Bs)):
                    ref.free_block(int(tables[b, j]))
                    tables[b, j] = -1
        torch.cuda.synchronize()
        assert np.array_equal(bt.cpu().numpy(), tables)
        assert B.pa_get_status() == 0
        assert _download_stack(h, stack) == [ref.allocate_block() for _ in range(ref.num_free())]
    finally:
        B.pa_pool_destroy(h)


@pytest.mark.parametrize("advance", ["torch", "step_call", "step_call_ahead"])
def test_device_loop_in_one_graph_matches_oracle(cuda_device, advance):
    """Workload-5-shaped loop (MHA, block 32) with every step on the device:
    pa_device_alloc_blocks -> pa_write_kv_and_decode -> lengths += 1, the
    whole run captured as one CUDA graph; against the host allocator + oracle.
    The lengths advance either by torch kernels or inside the allocation
    launch (pa_device_alloc_blocks_step, two length arrays taking turns), or
    that launch runs a step ahead on a second stream while the previous step
    decodes (three length arrays; it waits for the decode that last read the
    array it writes)."""
    import oracle
    from paged_kv_cache_239_gb300 import workloads as W
    from gpu_helpers import max_abs_err

    steps = 24
    wl = W.custom("devloop", "bf16", 1, 16, 16, 128, 32, [1, 31, 32, 33, 64, 95, 200, 7],
                  seed=8, steps=steps, spare_blocks=4)
    pool = W.make_pool(wl)
    ks, vs = W.make_new_tokens(wl, steps)
    qs = W.make_queries(wl, steps)
    pool_d = pool.to(cuda_device)
    h = B.pa_pool_create(pool_d, wl.num_blocks, 1, 16, 32, 128, pool_d.dtype)
    try:
        used = sorted(int(x) for x in wl.block_tables[wl.block_tables >= 0])
        order = list(wl.free_stack) + used
        B.pa_pool_seed_free_stack(h, order)
        for _ in used:
            B.pa_alloc_block(h)
        ref = FreeBlockStack(wl.num_blocks)
        ref.seed(order)
        for _ in used:
            ref.allocate_block()
        stack = torch.empty(wl.num_blocks + 1, dtype=torch.int32, device=cuda_device)
        B.pa_device_stack_upload(h, stack)
        bt = torch.from_numpy(wl.block_tables.copy()).to(cuda_device)
        lens = torch.from_numpy(wl.context_lens.copy()).to(cuda_device)
        lens1 = torch.empty_like(lens)
        kd, vd, qd = ks.to(cuda_device), vs.to(cuda_device), qs.to(cuda_device)
        outs = torch.zeros((steps, wl.batch, 16, 128), dtype=torch.float32, device=cuda_device)
        pb = 1
        need = B.pa_decode_workspace_size(h, wl.batch, 16, wl.max_blocks, pb)
        ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
        B.pa_get_status()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        lens2 = torch.empty_like(lens)
        if advance == "step_call_ahead":
            side = torch.cuda.Stream()
            bufs = (lens, lens1, lens2)
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    side.wait_stream(s)
                    ev_alloc = [torch.cuda.Event() for _ in range(steps)]
                    ev_dec = [torch.cuda.Event() for _ in range(steps)]

                    def alloc(t):
                        with torch.cuda.stream(side):
                            if t >= 2:
                                side.wait_event(ev_dec[t - 2])
                            B.pa_device_alloc_blocks_step(h, stack, bt, wl.max_blocks,
                                                          bufs[t % 3], bufs[(t + 1) % 3],
                                                          wl.batch, stream=side)
                            ev_alloc[t].record(side)

                    alloc(0)
                    for t in range(steps):
                        if t + 1 < steps:
                            alloc(t + 1)
                        s.wait_event(ev_alloc[t])
                        B.pa_write_kv_and_decode(outs[t], qd[t], h, 0, kd[t], vd[t],
                                                 bufs[t % 3], bt, wl.max_blocks,
                                                 bufs[(t + 1) % 3], wl.batch, 32, 16, 16, 128,
                                                 wl.scale, pb, ws, need, stream=s)
                        ev_dec[t].record(s)
                    s.wait_stream(side)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s) if advance != "step_call_ahead" else _null():
                for t in range(steps if advance != "step_call_ahead" else 0):
                    if advance == "torch":
                        cur, nxt = lens, lens1
                        B.pa_device_alloc_blocks(h, stack, bt, wl.max_blocks, cur, wl.batch,
                                                 stream=s)
                        torch.add(cur, 1, out=nxt)
                    else:
                        cur, nxt = (lens, lens1) if t % 2 == 0 else (lens1, lens)
                        B.pa_device_alloc_blocks_step(h, stack, bt, wl.max_blocks, cur, nxt,
                                                      wl.batch, stream=s)
                    B.pa_write_kv_and_decode(outs[t], qd[t], h, 0, kd[t], vd[t], cur, bt,
                                             wl.max_blocks, nxt, wl.batch, 32, 16, 16, 128,
                                             wl.scale, pb, ws, need, stream=s)
                    if advance == "torch":
                        lens.copy_(lens1)
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        # host reference of the same loop
        host = W.as_oracle_array(pool).copy()
        tables = wl.block_tables.copy()
        ln = wl.context_lens.copy()
        for t in range(steps):
            for b in range(wl.batch):
                if ln[b] % 32 == 0:
                    tables[b, ln[b] // 32] = ref.allocate_block()
            oracle.write_kv(host, 0, W.as_oracle_array(ks[t]), W.as_oracle_array(vs[t]), tables, ln)
            ln = ln + 1
            if t in (0, 1, steps - 1):
                r = oracle.decode_attention(W.as_oracle_array(qs[t]), host, 0, tables, ln, 16,
                                            wl.scale)
                assert max_abs_err(outs[t], r) <= 2e-3, t
        assert np.array_equal(bt.cpu().numpy(), tables)
        if advance == "step_call_ahead":
            final = (lens, lens1, lens2)[steps % 3]
        else:
            final = lens if (advance == "torch" or steps % 2 == 0) else lens1
        assert np.array_equal(final.cpu().numpy(), ln)
        assert np.array_equal(W.as_oracle_array(pool_d), host)
        assert B.pa_get_status() == 0
        assert _download_stack(h, stack) == [ref.allocate_block() for _ in range(ref.num_free())]
    finally:
        B.pa_pool_destroy(h)


def test_alloc_step_writes_next_lengths_and_refuses_overlap(cuda_device):
    """pa_device_alloc_blocks_step allocates exactly as pa_device_alloc_blocks
    and writes positions + 1; next_lens overlapping positions is refused before
    any launch."""
    nb, Bs, maxb = 12, 16, 4
    pool = torch.zeros((nb, 2, 1, 1, Bs, 64), dtype=torch.bfloat16, device=cuda_device)
    h = B.pa_pool_create(pool, nb, 1, 1, Bs, 64, pool.dtype)
    try:
        order = [int(x) for x in np.random.default_rng(3).permutation(nb)]
        B.pa_pool_seed_free_stack(h, order)
        stack = torch.empty(nb + 1, dtype=torch.int32, device=cuda_device)
        B.pa_device_stack_upload(h, stack)
        bt = torch.full((5, maxb), -1, dtype=torch.int32, device=cuda_device)
        pos = torch.tensor([0, 16, 5, 63, 32], dtype=torch.int32, device=cuda_device)
        nxt = torch.full((5,), -7, dtype=torch.int32, device=cuda_device)
        with pytest.raises(B.PagedAttnError) as e:
            B.pa_device_alloc_blocks_step(h, stack, bt, maxb, pos, pos, 5)
        assert e.value.code == B.PA_ERR_INVALID_ARG
        B.pa_device_alloc_blocks_step(h, stack, bt, maxb, pos, nxt, 5)
        torch.cuda.synchronize()
        assert nxt.cpu().tolist() == [1, 17, 6, 64, 33]
        ref = FreeBlockStack(nb)
        ref.seed(order)
        want = np.full((5, maxb), -1, dtype=np.int32)
        for b, p_ in enumerate([0, 16, 5, 63, 32]):
            if p_ % Bs == 0:
                want[b, p_ // Bs] = ref.allocate_block()
        assert np.array_equal(bt.cpu().numpy(), want)
        assert B.pa_get_status() == 0
        assert _download_stack(h, stack) == [ref.allocate_block() for _ in range(ref.num_free())]
    finally:
        B.pa_pool_destroy(h)
