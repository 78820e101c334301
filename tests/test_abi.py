"""The C ABI on the host (no GPU): the library loads, exports every function
the header declares, the allocator matches the oracle's free stack, and host-side
argument checks return the documented codes without touching a device."""
import ctypes
import subprocess

import numpy as np
import pytest

from oracle.allocator import FreeBlockStack

FAKE_DEV_PTR = 0x7F0000000000  # 16-byte aligned; never dereferenced by host-only calls


def test_every_header_symbol_is_exported(pa_lib):
    names = pa_lib.header_symbols()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", pa_lib.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    lib = pa_lib.lib()
    for n in names:
        assert getattr(lib, n) is not None


def test_only_header_functions_are_exported(pa_lib):
    """Internal symbols (kernels, launchers, the bundled CUDA runtime) are hidden,
    so two builds loaded in one process cannot interpose on each other."""
    out = subprocess.run(["nm", "-D", "--defined-only", pa_lib.library_path()],
                         capture_output=True, text=True, check=True).stdout
    funcs = [line.split()[-1] for line in out.splitlines() if " T " in line]
    assert sorted(funcs) == pa_lib.header_symbols()


def test_every_declaration_cites_its_passage():
    """Each exported call's comment names the page and section it restates, or
    says that the pages have no counterpart ("Cites:")."""
    import os

    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                        "pagedattn.h")
    lines = open(path).read().split("\n")
    missing = []
    for i, line in enumerate(lines):
        if not line.startswith("PA_API"):
            continue
        j = i - 1
        while j >= 0 and not lines[j].rstrip().endswith("*/"):
            j -= 1
        k = j
        while k >= 0 and "/*" not in lines[k]:
            k -= 1
        if "Cites:" not in "\n".join(lines[k:j + 1]):
            missing.append(line.split("(")[0].split()[-1])
    assert not missing, f"declarations without a citation: {missing}"


def _pool(pa_lib, nb=8, L=2, Hkv=2, B=16, D=64, dtype=1):
    return pa_lib.pa_pool_create(FAKE_DEV_PTR, nb, L, Hkv, B, D, dtype)


def test_allocator_matches_oracle_free_stack(pa_lib):
    h = _pool(pa_lib, nb=32)
    ref = FreeBlockStack(32)
    rng = np.random.default_rng(1)
    held = []
    try:
        for _ in range(3000):
            if held and (rng.random() < 0.5 or ref.num_free() == 0):
                b = held.pop(int(rng.integers(len(held))))
                pa_lib.pa_free_block(h, b)
                ref.free_block(b)
            else:
                a = pa_lib.pa_alloc_block(h)
                assert a == ref.allocate_block()
                held.append(a)
            assert pa_lib.pa_num_free(h) == ref.num_free()
    finally:
        pa_lib.pa_pool_destroy(h)


def test_allocator_first_id_and_exhaustion(pa_lib):
    h = _pool(pa_lib, nb=3)
    try:
        assert [pa_lib.pa_alloc_block(h) for _ in range(3)] == [2, 1, 0]
        with pytest.raises(MemoryError, match="Out of KV-Cache Physical Blocks"):
            pa_lib.pa_alloc_block(h)
        with pytest.raises(pa_lib.PagedAttnError) as e:
            pa_lib.pa_free_block(h, 3)
        assert e.value.code == pa_lib.PA_ERR_INVALID_ARG
        pa_lib.pa_free_block(h, 1)
        with pytest.raises(pa_lib.PagedAttnError) as e:
            pa_lib.pa_free_block(h, 1)
        assert e.value.code == pa_lib.PA_ERR_DOUBLE_FREE
        assert pa_lib.pa_alloc_block(h) == 1
    finally:
        pa_lib.pa_pool_destroy(h)


def test_seeded_free_stack_matches_oracle(pa_lib):
    order = list(np.random.default_rng(3).permutation(10))
    h = _pool(pa_lib, nb=10)
    ref = FreeBlockStack(10)
    ref.seed(order)
    try:
        pa_lib.pa_pool_seed_free_stack(h, order)
        assert [pa_lib.pa_alloc_block(h) for _ in range(10)] == [ref.allocate_block()
                                                                 for _ in range(10)]
        with pytest.raises(pa_lib.PagedAttnError):
            pa_lib.pa_pool_seed_free_stack(h, order)  # blocks in use
    finally:
        pa_lib.pa_pool_destroy(h)
    h = _pool(pa_lib, nb=4)
    try:
        with pytest.raises(pa_lib.PagedAttnError):
            pa_lib.pa_pool_seed_free_stack(h, [0, 1, 1, 2])
    finally:
        pa_lib.pa_pool_destroy(h)


def test_block_bytes(pa_lib):
    h = pa_lib.pa_pool_create(FAKE_DEV_PTR, 4, 24, 2, 16, 64, pa_lib.PA_DTYPE_BF16)
    try:
        assert pa_lib.pa_pool_block_bytes(h) == 196608
    finally:
        pa_lib.pa_pool_destroy(h)


@pytest.mark.parametrize("args", [
    (0, 8, 1, 1, 16, 64, 1),                 # NULL pool
    (FAKE_DEV_PTR + 8, 8, 1, 1, 16, 64, 1),  # misaligned
    (FAKE_DEV_PTR, 0, 1, 1, 16, 64, 1),      # no blocks
    (FAKE_DEV_PTR, 8, 1, 1, 16, 4, 1),       # row not a multiple of 16 bytes
    (FAKE_DEV_PTR, 8, 1, 1, 16, 64, 7),      # unknown dtype
])
def test_pool_create_rejects_bad_arguments(pa_lib, args):
    with pytest.raises(pa_lib.PagedAttnError) as e:
        pa_lib.pa_pool_create(*args)
    assert e.value.code == pa_lib.PA_ERR_INVALID_ARG


def test_decode_host_checks(pa_lib):
    h = _pool(pa_lib, nb=8, L=2, Hkv=2, B=16, D=64)
    F = FAKE_DEV_PTR
    try:
        def call(**kw):
            a = dict(out=F, q=F, pool=h, layer=0, bt=F, maxb=4, lens=F, batch=2, B=16, H=4,
                     Hkv=2, D=64, scale=0.125, pb=2, ws=None, wsb=0)
            a.update(kw)
            pa_lib.pa_decode_attention_partitioned(a["out"], a["q"], a["pool"], a["layer"], a["bt"],
                                                   a["maxb"], a["lens"], a["batch"], a["B"], a["H"],
                                                   a["Hkv"], a["D"], a["scale"], a["pb"], a["ws"],
                                                   a["wsb"], 0)

        for bad, code in [(dict(layer=2), 1), (dict(B=32), 1), (dict(Hkv=1), 1), (dict(D=128), 1),
                          (dict(H=5), 1), (dict(maxb=0), 1), (dict(pb=-1), 1),
                          (dict(scale=float("nan")), 1),
                          # groups of 9 and 17 are served (8-head chunks, the last
                          # ragged): the call fails only for want of a workspace
                          (dict(H=18), 6), (dict(H=34), 6),
                          (dict(ws=None, wsb=0), 6), (dict(ws=F + 64, wsb=1 << 30), 6),
                          (dict(ws=F, wsb=16), 6)]:
            with pytest.raises(pa_lib.PagedAttnError) as e:
                call(**bad)
            assert e.value.code == code, (bad, e.value)
        # batch 0 is a no-op that needs no device
        call(batch=0)
        # an fp32 pool runs only on the CUDA-core kernel (any group: a group of
        # 3 fails only for want of a workspace); the tensor-core kernels refuse it
        h32 = _pool(pa_lib, nb=8, L=2, Hkv=2, B=16, D=64, dtype=0)
        try:
            with pytest.raises(pa_lib.PagedAttnError) as e:
                call(pool=h32, H=6)
            assert e.value.code == pa_lib.PA_ERR_WORKSPACE
            pa_lib.pa_pool_set_decode_kernel(h32, pa_lib.PA_DECODE_TENSOR_CORES)
            with pytest.raises(pa_lib.PagedAttnError) as e:
                call(pool=h32, H=6)
            assert e.value.code == pa_lib.PA_ERR_UNSUPPORTED
        finally:
            pa_lib.pa_pool_destroy(h32)
        with pytest.raises(pa_lib.PagedAttnError) as e:
            call(out=F + 4, ws=F, wsb=1 << 20)
        assert e.value.code == pa_lib.PA_ERR_INVALID_ARG
    finally:
        pa_lib.pa_pool_destroy(h)


def test_workspace_size_formula(pa_lib):
    h = _pool(pa_lib, nb=8, L=1, Hkv=2, B=16, D=64)
    try:
        # maxb 10 blocks, 3 per partition -> 4 partitions
        got = pa_lib.pa_decode_workspace_size(h, 5, 8, 10, 3)
        slots = 5 * 8 * 4
        assert got == ((slots * 64 * 4 + 255) // 256) * 256 + slots * 2 * 4
        assert pa_lib.pa_decode_workspace_size(h, 5, 8, 10, 10) == 0
        assert pa_lib.pa_decode_workspace_size(h, 5, 8, 10, 64) == 0
    finally:
        pa_lib.pa_pool_destroy(h)


def test_write_kv_and_gather_host_checks(pa_lib):
    h = _pool(pa_lib)
    F = FAKE_DEV_PTR
    try:
        pa_lib.pa_write_kv(h, 0, F, F, F, 4, F, 0, 0)  # batch 0: no-op
        for args in [(h, 2, F, F, F, 4, F, 1, 0), (h, 0, F + 8, F, F, 4, F, 1, 0),
                     (h, 0, None, F, F, 4, F, 1, 0), (h, 0, F, F, F, 0, F, 1, 0)]:
            with pytest.raises(pa_lib.PagedAttnError) as e:
                pa_lib.pa_write_kv(*args)
            assert e.value.code == pa_lib.PA_ERR_INVALID_ARG
        pa_lib.pa_gather_kv(F, F, F, h, 0, F, 4, F, 3, 0, 0)  # max_len 0: no-op
        with pytest.raises(pa_lib.PagedAttnError):
            pa_lib.pa_gather_kv(F + 4, F, F, h, 0, F, 4, F, 3, 10, 0)
    finally:
        pa_lib.pa_pool_destroy(h)


def test_null_handle_and_error_string(pa_lib):
    with pytest.raises(pa_lib.PagedAttnError):
        pa_lib.pa_num_free(None)
    assert "NULL" in pa_lib.last_error()
    pa_lib.pa_pool_destroy(None)
    assert isinstance(ctypes.c_int(pa_lib.PA_OK).value, int)


def test_strided_pool_checks(pa_lib):
    F = FAKE_DEV_PTR
    D, Bs, Hkv, L, nb = 64, 16, 2, 3, 10
    tile = Bs * D
    ok = [(F, F + (1 << 30), Hkv * tile, 0, tile, nb, 1, Hkv),      # separate K / V caches, 1 layer
          (F, F + (1 << 30), Hkv * tile, nb * Hkv * tile, tile, nb, L, Hkv)]  # layer-major stack
    for kb, vb, sb, sl, sh, n, layers, heads in ok:
        h = pa_lib.pa_pool_create_strided(kb, vb, sb, sl, sh, n, layers, heads, Bs, D, 1)
        pa_lib.pa_pool_destroy(h)
    bad = [(F + 8, F, Hkv * tile, 0, tile, nb, 1, Hkv),          # misaligned base
           (F, F, Hkv * tile, 0, tile // 2, nb, 1, Hkv),          # heads overlap
           (F, F, tile, 0, tile, nb, 1, Hkv),                     # blocks overlap heads
           (F, F, Hkv * tile, 0, tile, nb, 2, Hkv),               # zero stride, two layers
           (F, F, Hkv * tile + 1, 0, tile, nb, 1, Hkv),           # stride not 16-byte multiple
           (F, F, -Hkv * tile, 0, tile, nb, 1, Hkv),              # negative
           (F, None, Hkv * tile, 0, tile, nb, 1, Hkv)]            # NULL V base
    for args in bad:
        with pytest.raises(pa_lib.PagedAttnError) as e:
            pa_lib.pa_pool_create_strided(*args, Bs, D, 1)
        assert e.value.code == pa_lib.PA_ERR_INVALID_ARG, args


def test_decode_kernel_choice_query(pa_lib):
    """Which kernel a call runs (host only): automatic choice by dtype, head_dim
    and group; forced kinds that cannot serve the shape are refused."""
    L = pa_lib
    cases = [  # (Hkv, D, dtype, num_heads, automatic kernel)
        (2, 64, 1, 16, L.PA_DECODE_TENSOR_CORES),    # bf16, group 8
        (2, 128, 1, 8, L.PA_DECODE_TENSOR_CORES),    # bf16, group 4
        (1, 128, 1, 16, L.PA_DECODE_TCGEN05),        # bf16, head_dim 128, group 16
        (2, 128, 1, 128, L.PA_DECODE_TCGEN05),       # group 64
        (1, 128, 1, 24, L.PA_DECODE_TENSOR_CORES),   # group 24: not a multiple of 16
        (1, 128, 1, 71, L.PA_DECODE_TENSOR_CORES),   # group 71: 8-head chunks, the last of 7
        (8, 128, 1, 232, L.PA_DECODE_TENSOR_CORES),  # group 29
        (1, 128, 1, 128, L.PA_DECODE_TCGEN05),       # group 128: one chunk, heads on the rows
        (1, 64, 1, 32, L.PA_DECODE_TENSOR_CORES),    # head_dim 64: no tcgen05
        (2, 64, 0, 8, L.PA_DECODE_CUDA_CORES),       # fp32
    ]
    for Hkv, D, dtype, H, want in cases:
        h = _pool(pa_lib, Hkv=Hkv, D=D, dtype=dtype)
        try:
            assert L.pa_decode_kernel_choice(h, H) == want, (Hkv, D, dtype, H)
            # the CUDA-core kernel serves every group (power-of-two head chunks,
            # the heads past the group masked)
            L.pa_pool_set_decode_kernel(h, L.PA_DECODE_CUDA_CORES)
            assert L.pa_decode_kernel_choice(h, H) == L.PA_DECODE_CUDA_CORES
            L.pa_pool_set_decode_kernel(h, L.PA_DECODE_TCGEN05)
            if want == L.PA_DECODE_TCGEN05:
                assert L.pa_decode_kernel_choice(h, H) == L.PA_DECODE_TCGEN05
            else:
                with pytest.raises(L.PagedAttnError) as e:
                    L.pa_decode_kernel_choice(h, H)
                assert e.value.code == L.PA_ERR_UNSUPPORTED
            with pytest.raises(L.PagedAttnError) as e:
                L.pa_decode_kernel_choice(h, H + 1 if Hkv > 1 else 0)
            assert e.value.code == L.PA_ERR_INVALID_ARG
        finally:
            L.pa_pool_destroy(h)


def test_decode_kernel_choice_checks(pa_lib):
    h = _pool(pa_lib)
    try:
        for kind in (pa_lib.PA_DECODE_AUTO, pa_lib.PA_DECODE_CUDA_CORES,
                     pa_lib.PA_DECODE_TENSOR_CORES, pa_lib.PA_DECODE_TCGEN05):
            pa_lib.pa_pool_set_decode_kernel(h, kind)
        with pytest.raises(pa_lib.PagedAttnError) as e:
            pa_lib.pa_pool_set_decode_kernel(h, 4)
        assert e.value.code == pa_lib.PA_ERR_INVALID_ARG
    finally:
        pa_lib.pa_pool_destroy(h)
