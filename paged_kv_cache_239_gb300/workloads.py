"""Seeded synthetic workloads shaped like the source pages' examples.

This module only draws inputs: context lengths, block tables popped from a
shuffled free-block stack, and N(0,1) values for the pool, queries and new
tokens.  It contains none of the attention or slot-resolution arithmetic, and
it is the one module that both the CUDA path's tests/benchmark and the CPU
oracle's checks take their inputs from.

The five named workloads (numbers are the seeds' offsets from 239):
  1 tiny_f32                 fp32, 1 layer, batch 2, 2 heads / 2 KV heads,
                             head_dim 64, block 16, lengths {17, 40}, 8 blocks,
                             tables from a seeded permutation of 0..7, scale 1/8.
  2 mini_infer_bf16          bf16 pool [nb, 2, 24, 2, 16, 64] (the mini-infer
                             BlockPool defaults), 16 query heads (group 8),
                             batch 32, lengths U[16, 800], pool = 1.1x the
                             blocks needed, tables popped from a shuffled stack.
  3 large_batch_bf16         bf16, batch 256, 32 heads / 8 KV heads, head_dim 128,
                             block 16, 32 layers, lengths U[128, 4096], blocks
                             popped round-robin across sequences (interleaved).
  4 long_context_bf16        bf16, batch 4, 32 / 8 heads, head_dim 128, block 32,
                             1 layer, lengths {32768, 65536, 100000, 131072},
                             random block permutation (split-K workload).
  5 append_decode_loop_bf16  bf16 MHA, batch 64, 32 heads, head_dim 128, block 32,
                             1 layer, start lengths U[1, 1024] with {1, 31, 32, 33,
                             64, 1024} forced, 64 append+decode steps.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

SEED_BASE = 239

NAMES = {
    1: "tiny_f32",
    2: "mini_infer_bf16",
    3: "large_batch_bf16",
    4: "long_context_bf16",
    5: "append_decode_loop_bf16",
}


@dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    num_layers: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    context_lens: np.ndarray   # int32 [batch]
    block_tables: np.ndarray   # int32 [batch, max_blocks], -1 where unused
    num_blocks: int
    scale: float
    seed: int
    free_stack: List[int] = field(default_factory=list)  # ids still free; pop() from the end
    steps: int = 0             # append+decode steps (workload 5)

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def pool_shape(self):
        return (self.num_blocks, 2, self.num_layers, self.num_kv_heads, self.block_size,
                self.head_dim)

    def pool_bytes(self) -> int:
        return int(np.prod(self.pool_shape())) * self.elem_bytes


def _ceil_div(a, b):
    return -(-a // b)


def _pop_tables(lens: np.ndarray, block_size: int, max_blocks: int, stack: List[int],
                interleave: bool) -> np.ndarray:
    nblk = [_ceil_div(int(n), block_size) for n in lens]
    tables = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    if interleave:
        for j in range(max(nblk) if nblk else 0):
            for b, nb in enumerate(nblk):
                if j < nb:
                    tables[b, j] = stack.pop()
    else:
        for b, nb in enumerate(nblk):
            for j in range(nb):
                tables[b, j] = stack.pop()
    return tables


def custom(name: str, dtype: str, num_layers: int, num_heads: int, num_kv_heads: int,
           head_dim: int, block_size: int, lens, seed: int, spare_blocks: int = 0,
           interleave: bool = False, max_blocks: Optional[int] = None,
           scale: Optional[float] = None, steps: int = 0) -> Workload:
    """A workload with the given lengths; tables popped from a shuffled stack."""
    lens = np.asarray(lens, dtype=np.int32)
    rng = np.random.default_rng(seed)
    need_lens = lens + steps
    need = int(sum(_ceil_div(int(n), block_size) for n in need_lens))
    nb = max(1, need + spare_blocks)
    if max_blocks is None:
        max_blocks = max(1, max(_ceil_div(int(n), block_size) for n in need_lens) if len(lens) else 1)
    stack = [int(x) for x in rng.permutation(nb)]
    tables = _pop_tables(lens, block_size, max_blocks, stack, interleave)
    return Workload(name, dtype, num_layers, num_heads, num_kv_heads, head_dim, block_size, lens,
                    tables, nb, scale if scale is not None else 1.0 / math.sqrt(head_dim), seed,
                    stack, steps)


def named(cfg: int) -> Workload:
    """One of the five named workloads (1..5)."""
    seed = SEED_BASE + cfg
    rng = np.random.default_rng(seed)
    if cfg == 1:
        lens = np.array([17, 40], dtype=np.int32)
        perm = [int(x) for x in rng.permutation(8)]
        tables = np.full((2, 3), -1, dtype=np.int32)
        tables[0, :2] = perm[0:2]
        tables[1, :3] = perm[2:5]
        return Workload(NAMES[1], "f32", 1, 2, 2, 64, 16, lens, tables, 8, 1.0 / 8.0, seed,
                        perm[5:][::-1])
    if cfg == 2:
        lens = rng.integers(16, 801, size=32).astype(np.int32)
        need = int(sum(_ceil_div(int(n), 16) for n in lens))
        nb = math.ceil(1.1 * need)
        stack = [int(x) for x in rng.permutation(nb)]
        tables = _pop_tables(lens, 16, _ceil_div(800, 16), stack, interleave=False)
        return Workload(NAMES[2], "bf16", 24, 16, 2, 64, 16, lens, tables, nb, 1.0 / 8.0, seed,
                        stack)
    if cfg == 3:
        lens = rng.integers(128, 4097, size=256).astype(np.int32)
        need = int(sum(_ceil_div(int(n), 16) for n in lens))
        nb = need + 256
        stack = [int(x) for x in rng.permutation(nb)]
        tables = _pop_tables(lens, 16, 4096 // 16, stack, interleave=True)
        return Workload(NAMES[3], "bf16", 32, 32, 8, 128, 16, lens, tables, nb,
                        1.0 / math.sqrt(128), seed, stack)
    if cfg == 4:
        lens = np.array([32768, 65536, 100000, 131072], dtype=np.int32)
        need = int(sum(_ceil_div(int(n), 32) for n in lens))
        stack = [int(x) for x in rng.permutation(need)]
        tables = _pop_tables(lens, 32, 131072 // 32, stack, interleave=False)
        return Workload(NAMES[4], "bf16", 1, 32, 8, 128, 32, lens, tables, need,
                        1.0 / math.sqrt(128), seed, stack)
    if cfg == 5:
        steps = 64
        lens = rng.integers(1, 1025, size=64).astype(np.int32)
        lens[:6] = [1, 31, 32, 33, 64, 1024]
        need = int(sum(_ceil_div(int(n) + steps, 32) for n in lens))
        nb = math.ceil(1.1 * need)
        stack = [int(x) for x in rng.permutation(nb)]
        tables = _pop_tables(lens, 32, _ceil_div(1024 + steps, 32), stack, interleave=False)
        return Workload(NAMES[5], "bf16", 1, 32, 32, 128, 32, lens, tables, nb,
                        1.0 / math.sqrt(128), seed, stack, steps)
    raise ValueError(f"unknown workload {cfg}")


# ------------------------------------------------------------------ values


def torch_dtype(wl: Workload):
    import torch

    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def _gen(device, seed: int):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_pool(wl: Workload, device="cpu", seed_offset: int = 0, chunk_bytes: int = 1 << 30):
    """The pool tensor filled with N(0,1) values (drawn in fp32, cast to the dtype)."""
    import torch

    dt = torch_dtype(wl)
    pool = torch.empty(wl.pool_shape(), dtype=dt, device=device)
    g = _gen(device, wl.seed * 1000 + 1 + seed_offset)
    per_block = int(np.prod(wl.pool_shape()[1:])) * 4
    cb = max(1, chunk_bytes // per_block)
    for i in range(0, wl.num_blocks, cb):
        j = min(wl.num_blocks, i + cb)
        tmp = torch.randn((j - i,) + wl.pool_shape()[1:], generator=g, device=device,
                          dtype=torch.float32)
        pool[i:j].copy_(tmp)
        del tmp
    return pool


def make_queries(wl: Workload, count: int, device="cpu", seed_offset: int = 0):
    """`count` query batches [count, batch, num_heads, head_dim] of N(0,1)."""
    import torch

    g = _gen(device, wl.seed * 1000 + 2 + seed_offset)
    q = torch.randn((count, wl.batch, wl.num_heads, wl.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch_dtype(wl))


def make_new_tokens(wl: Workload, count: int, device="cpu", seed_offset: int = 0):
    """`count` new-token K and V batches, each [count, batch, num_kv_heads, head_dim]."""
    import torch

    g = _gen(device, wl.seed * 1000 + 3 + seed_offset)
    shape = (count, wl.batch, wl.num_kv_heads, wl.head_dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return k.to(torch_dtype(wl)), v.to(torch_dtype(wl))


def as_oracle_array(t):
    """A CPU numpy view of a tensor in the oracle's element convention
    (float32 stays float32; bf16 becomes its raw uint16 bit patterns)."""
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
