"""CPU oracle for paged KV-cache decode attention, KV append and batched gather.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  The
product library (``paged_kv_cache_239_gb300``) never imports, links or runs
anything here, and this package never imports the product library: the two
share no code.

Contents
--------
``pa_oracle.c``   fp64 decode attention, KV append and batched gather in plain C
                  (OpenMP over sequences and heads), compiled by :func:`build`.
``allocator``     the free-block stack of the mini-infer BlockPool.
``waste``         last-block internal-fragmentation arithmetic.
``brute``         a second, NumPy-only decode attention for tiny inputs.

Every function cites the passage of the source pages it follows; see the
header of ``pa_oracle.c`` for the attention and append definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpa_oracle.so")

F32 = 0
BF16 = 1

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` with gcc into ``oracle/_build/libpa_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_decode_attention.argtypes = [P, P, P, I, I, I, I, I, I, I, P, I, P, I, I, D, I]
        lib.oracle_decode_attention.restype = I
        lib.oracle_write_kv.argtypes = [P, I, I, I, I, I, I, I, P, P, P, I, P, I]
        lib.oracle_write_kv.restype = I
        lib.oracle_gather_kv.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, I, P, I, I]
        lib.oracle_gather_kv.restype = I
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP loop uses by default on this host."""
    return int(_load().oracle_max_threads())


def _raw(a: np.ndarray) -> np.ndarray:
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle inputs must be C-contiguous")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dtype_code(arr: np.ndarray) -> int:
    """float32 arrays are fp32; uint16 arrays carry raw bf16 bit patterns."""
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"pool/q must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def decode_attention(q: np.ndarray, pool: np.ndarray, layer: int, block_tables,
                     context_lens, num_heads: int, scale: float,
                     threads: Optional[int] = None) -> np.ndarray:
    """fp64 paged decode attention.

    ``pool`` has shape [num_blocks, 2, L, Hkv, B, D] (float32, or uint16 holding bf16
    bits); ``q`` is [batch, num_heads, D] of the same element type; ``block_tables``
    is int32 [batch, max_blocks]; ``context_lens`` int32 [batch].  Returns fp64
    [batch, num_heads, D].  Follows the definition in ``pa_oracle.c``.
    """
    pool = _raw(pool)
    q = _raw(q)
    dt = _dtype_code(pool)
    if _dtype_code(q) != dt:
        raise TypeError("q and pool must share one element type")
    nb, two, L, Hkv, B, D = pool.shape
    assert two == 2
    bt = _i32(block_tables)
    lens = _i32(context_lens)
    batch = lens.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == batch
    assert q.shape == (batch, num_heads, D)
    out = np.zeros((batch, num_heads, D), dtype=np.float64)
    nthr = threads if threads is not None else max_threads()
    rc = _load().oracle_decode_attention(
        out.ctypes.data, q.ctypes.data, pool.ctypes.data, dt, nb, L, Hkv, B, D, layer,
        bt.ctypes.data, bt.shape[1], lens.ctypes.data, batch, num_heads, float(scale), nthr)
    if rc != 0:
        raise ValueError(f"oracle_decode_attention rejected its arguments (rc={rc})")
    return out


def write_kv(pool: np.ndarray, layer: int, k: np.ndarray, v: np.ndarray, block_tables,
             positions) -> None:
    """Append one token per sequence in place: K/V rows to slot (bt[p/B], p%B)."""
    pool = _raw(pool)
    dt = _dtype_code(pool)
    nb, _, L, Hkv, B, D = pool.shape
    k = _raw(k)
    v = _raw(v)
    bt = _i32(block_tables)
    pos = _i32(positions)
    batch = pos.shape[0]
    assert k.shape == (batch, Hkv, D) and v.shape == (batch, Hkv, D)
    assert k.dtype == pool.dtype and v.dtype == pool.dtype
    rc = _load().oracle_write_kv(pool.ctypes.data, dt, nb, L, Hkv, B, D, layer, k.ctypes.data,
                                 v.ctypes.data, bt.ctypes.data, bt.shape[1], pos.ctypes.data,
                                 batch)
    if rc != 0:
        raise ValueError(f"oracle_write_kv rejected its arguments (rc={rc})")


def gather_kv(pool: np.ndarray, layer: int, block_tables, context_lens, max_len: int):
    """Contiguous [batch, max_len, Hkv, D] K and V plus a bool mask (True = valid)."""
    pool = _raw(pool)
    dt = _dtype_code(pool)
    nb, _, L, Hkv, B, D = pool.shape
    bt = _i32(block_tables)
    lens = _i32(context_lens)
    batch = lens.shape[0]
    k_out = np.empty((batch, max_len, Hkv, D), dtype=pool.dtype)
    v_out = np.empty((batch, max_len, Hkv, D), dtype=pool.dtype)
    mask = np.empty((batch, max_len), dtype=np.uint8)
    rc = _load().oracle_gather_kv(k_out.ctypes.data, v_out.ctypes.data, mask.ctypes.data,
                                  pool.ctypes.data, dt, nb, L, Hkv, B, D, layer, bt.ctypes.data,
                                  bt.shape[1], lens.ctypes.data, batch, max_len)
    if rc != 0:
        raise ValueError(f"oracle_gather_kv rejected its arguments (rc={rc})")
    return k_out, v_out, mask.astype(bool)


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns (uint16) to float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
