"""ctypes binding of ``libpagedattn.so`` -- argument marshalling only.

Every function keeps the name of the C entry point it wraps (``include/pagedattn.h``)
and accepts torch tensors (their ``data_ptr()`` is passed), plain integers
(device addresses) or ``None`` (NULL).  Streams default to torch's current CUDA
stream.  All computation happens in the library's CUDA kernels; this module
never falls back to anything else, and raises if the library is not built.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

from ._build_lib import LIB_PATH, INCLUDE

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_NO_FREE_BLOCKS = 2
PA_ERR_DOUBLE_FREE = 3
PA_ERR_CUDA = 4
PA_ERR_UNSUPPORTED = 5
PA_ERR_WORKSPACE = 6

PA_DECODE_AUTO = 0
PA_DECODE_CUDA_CORES = 1
PA_DECODE_TENSOR_CORES = 2
PA_DECODE_TCGEN05 = 3

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1

PA_STATUS_BAD_BLOCK_ID = 0x1
PA_STATUS_BAD_LENGTH = 0x2
PA_STATUS_TIMEOUT = 0x4
PA_STATUS_NO_FREE_BLOCKS = 0x8

_ERR_NAMES = {
    PA_ERR_INVALID_ARG: "PA_ERR_INVALID_ARG",
    PA_ERR_NO_FREE_BLOCKS: "PA_ERR_NO_FREE_BLOCKS",
    PA_ERR_DOUBLE_FREE: "PA_ERR_DOUBLE_FREE",
    PA_ERR_CUDA: "PA_ERR_CUDA",
    PA_ERR_UNSUPPORTED: "PA_ERR_UNSUPPORTED",
    PA_ERR_WORKSPACE: "PA_ERR_WORKSPACE",
}


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, func: str, message: str):
        super().__init__(f"{func} failed with {_ERR_NAMES.get(code, code)}: {message}")
        self.code = code


class OutOfBlocksError(PagedAttnError, MemoryError):
    """Raised when the free-block stack is exhausted."""


_lib: Optional[ctypes.CDLL] = None


class pa_pool_layout(ctypes.Structure):
    """Mirror of the C struct: K/V base addresses and element strides."""
    _fields_ = [("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p),
                ("block_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64)]

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_PI = ctypes.POINTER(ctypes.c_int)
_PSZ = ctypes.POINTER(ctypes.c_size_t)
_PU = ctypes.POINTER(ctypes.c_uint)

_SIGNATURES = {
    "pa_last_error_string": ([], ctypes.c_char_p),
    "pa_pool_create": ([ctypes.POINTER(_P), _P, _I, _I, _I, _I, _I, _I], _I),
    "pa_pool_create_strided": ([ctypes.POINTER(_P), ctypes.POINTER(pa_pool_layout), _I, _I, _I,
                                _I, _I, _I], _I),
    "pa_pool_destroy": ([_P], _I),
    "pa_pool_block_bytes": ([_P, _PSZ], _I),
    "pa_pool_set_decode_kernel": ([_P, _I], _I),
    "pa_decode_kernel_choice": ([_P, _I, _PI], _I),
    "pa_pool_seed_free_stack": ([_P, _P, _I], _I),
    "pa_alloc_block": ([_P, _PI], _I),
    "pa_free_block": ([_P, _I], _I),
    "pa_num_free": ([_P, _PI], _I),
    "pa_write_kv": ([_P, _I, _P, _P, _P, _I, _P, _I, _P], _I),
    "pa_device_stack_bytes": ([_P, _PSZ], _I),
    "pa_device_stack_upload": ([_P, _P, _P], _I),
    "pa_device_stack_download": ([_P, _P, _P], _I),
    "pa_device_alloc_blocks": ([_P, _P, _P, _I, _P, _I, _P], _I),
    "pa_device_alloc_blocks_step": ([_P, _P, _P, _I, _P, _P, _I, _P], _I),
    "pa_device_free_blocks": ([_P, _P, _P, _I, _P, _P, _I, _P], _I),
    "pa_decode_attention": ([_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P], _I),
    "pa_decode_attention_partitioned": (
        [_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P], _I),
    "pa_write_kv_and_decode": ([_P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _F,
                                _I, _P, _SZ, _P], _I),
    "pa_decode_partition_blocks": ([_P, _I, _I, _I, _PI], _I),
    "pa_decode_workspace_size": ([_P, _I, _I, _I, _I, _PSZ], _I),
    "pa_decode_attention_noalloc": (
        [_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "pa_gather_kv": ([_P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P], _I),
    "pa_get_status": ([_PU, _P], _I),
    "pa_selftest_wait_timeout": ([_P], _I),
}


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or python -m paged_kv_cache_239_gb300._build_lib)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def header_symbols() -> list:
    """Names of the functions declared in include/pagedattn.h."""
    text = open(os.path.join(INCLUDE, "pagedattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def last_error() -> str:
    return lib().pa_last_error_string().decode()


def _check(rc: int, func: str) -> None:
    if rc != PA_OK:
        msg = last_error()
        if rc == PA_ERR_NO_FREE_BLOCKS:
            raise OutOfBlocksError(rc, func, msg)
        raise PagedAttnError(rc, func, msg)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    dp = getattr(x, "data_ptr", None)
    if dp is not None:
        return dp()
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    name = str(dtype)
    if name in ("torch.float32", "float32", "f32", "fp32"):
        return PA_DTYPE_F32
    if name in ("torch.bfloat16", "bfloat16", "bf16"):
        return PA_DTYPE_BF16
    raise ValueError(f"unsupported dtype {dtype}")


# --------------------------------------------------------------------- pool


def pa_pool_create(pool_dev, num_blocks: int, num_layers: int, num_kv_heads: int,
                   block_size: int, head_dim: int, dtype) -> int:
    h = _P()
    _check(lib().pa_pool_create(ctypes.byref(h), _ptr(pool_dev), num_blocks, num_layers,
                                num_kv_heads, block_size, head_dim, _dtype_code(dtype)),
           "pa_pool_create")
    return h.value


def pa_pool_create_strided(k_base, v_base, block_stride: int, layer_stride: int,
                           head_stride: int, num_blocks: int, num_layers: int, num_kv_heads: int,
                           block_size: int, head_dim: int, dtype) -> int:
    lay = pa_pool_layout(_ptr(k_base), _ptr(v_base), block_stride, layer_stride, head_stride)
    h = _P()
    _check(lib().pa_pool_create_strided(ctypes.byref(h), ctypes.byref(lay), num_blocks,
                                        num_layers, num_kv_heads, block_size, head_dim,
                                        _dtype_code(dtype)), "pa_pool_create_strided")
    return h.value


def pa_pool_destroy(pool: int) -> None:
    _check(lib().pa_pool_destroy(pool), "pa_pool_destroy")


def pa_pool_set_decode_kernel(pool: int, kind: int) -> None:
    _check(lib().pa_pool_set_decode_kernel(pool, kind), "pa_pool_set_decode_kernel")


def pa_decode_kernel_choice(pool: int, num_heads: int) -> int:
    v = ctypes.c_int()
    _check(lib().pa_decode_kernel_choice(pool, num_heads, ctypes.byref(v)),
           "pa_decode_kernel_choice")
    return v.value


def pa_pool_block_bytes(pool: int) -> int:
    v = _SZ()
    _check(lib().pa_pool_block_bytes(pool, ctypes.byref(v)), "pa_pool_block_bytes")
    return v.value


def pa_pool_seed_free_stack(pool: int, order) -> None:
    arr = (ctypes.c_int * len(order))(*[int(x) for x in order])
    _check(lib().pa_pool_seed_free_stack(pool, ctypes.cast(arr, _P), len(order)),
           "pa_pool_seed_free_stack")


def pa_alloc_block(pool: int) -> int:
    v = ctypes.c_int()
    _check(lib().pa_alloc_block(pool, ctypes.byref(v)), "pa_alloc_block")
    return v.value


def pa_free_block(pool: int, block_id: int) -> None:
    _check(lib().pa_free_block(pool, block_id), "pa_free_block")


def pa_num_free(pool: int) -> int:
    v = ctypes.c_int()
    _check(lib().pa_num_free(pool, ctypes.byref(v)), "pa_num_free")
    return v.value


# ------------------------------------------------------------ device stack


def pa_device_stack_bytes(pool: int) -> int:
    v = _SZ()
    _check(lib().pa_device_stack_bytes(pool, ctypes.byref(v)), "pa_device_stack_bytes")
    return v.value


def pa_device_stack_upload(pool: int, dev_stack, stream=None) -> None:
    _check(lib().pa_device_stack_upload(pool, _ptr(dev_stack), _stream(stream)),
           "pa_device_stack_upload")


def pa_device_stack_download(pool: int, dev_stack, stream=None) -> None:
    _check(lib().pa_device_stack_download(pool, _ptr(dev_stack), _stream(stream)),
           "pa_device_stack_download")


def pa_device_alloc_blocks(pool: int, dev_stack, block_tables, max_blocks_per_seq: int, positions,
                           batch: int, stream=None) -> None:
    _check(lib().pa_device_alloc_blocks(pool, _ptr(dev_stack), _ptr(block_tables),
                                        max_blocks_per_seq, _ptr(positions), batch,
                                        _stream(stream)), "pa_device_alloc_blocks")


def pa_device_alloc_blocks_step(pool: int, dev_stack, block_tables, max_blocks_per_seq: int,
                                positions, next_lens, batch: int, stream=None) -> None:
    _check(lib().pa_device_alloc_blocks_step(pool, _ptr(dev_stack), _ptr(block_tables),
                                             max_blocks_per_seq, _ptr(positions),
                                             _ptr(next_lens), batch, _stream(stream)),
           "pa_device_alloc_blocks_step")


def pa_device_free_blocks(pool: int, dev_stack, block_tables, max_blocks_per_seq: int,
                          context_lens, finished, batch: int, stream=None) -> None:
    _check(lib().pa_device_free_blocks(pool, _ptr(dev_stack), _ptr(block_tables),
                                       max_blocks_per_seq, _ptr(context_lens), _ptr(finished),
                                       batch, _stream(stream)), "pa_device_free_blocks")


# ---------------------------------------------------------------- kernels


def pa_write_kv(pool: int, layer: int, k, v, block_tables, max_blocks_per_seq: int, positions,
                batch: int, stream=None) -> None:
    _check(lib().pa_write_kv(pool, layer, _ptr(k), _ptr(v), _ptr(block_tables),
                             max_blocks_per_seq, _ptr(positions), batch, _stream(stream)),
           "pa_write_kv")


def pa_decode_partition_blocks(pool: int, batch: int, num_heads: int,
                               max_blocks_per_seq: int) -> int:
    v = ctypes.c_int()
    _check(lib().pa_decode_partition_blocks(pool, batch, num_heads, max_blocks_per_seq,
                                            ctypes.byref(v)), "pa_decode_partition_blocks")
    return v.value


def pa_decode_workspace_size(pool: int, batch: int, num_heads: int, max_blocks_per_seq: int,
                             partition_blocks: int = 0) -> int:
    v = _SZ()
    _check(lib().pa_decode_workspace_size(pool, batch, num_heads, max_blocks_per_seq,
                                          partition_blocks, ctypes.byref(v)),
           "pa_decode_workspace_size")
    return v.value


def pa_decode_attention(out, q, pool: int, layer: int, block_tables, max_blocks_per_seq: int,
                        context_lens, batch: int, block_size: int, num_heads: int,
                        num_kv_heads: int, head_dim: int, scale: float, workspace=None,
                        workspace_bytes: int = 0, stream=None) -> None:
    _check(lib().pa_decode_attention(_ptr(out), _ptr(q), pool, layer, _ptr(block_tables),
                                     max_blocks_per_seq, _ptr(context_lens), batch, block_size,
                                     num_heads, num_kv_heads, head_dim, float(scale),
                                     _ptr(workspace), workspace_bytes, _stream(stream)),
           "pa_decode_attention")


def pa_decode_attention_partitioned(out, q, pool: int, layer: int, block_tables,
                                    max_blocks_per_seq: int, context_lens, batch: int,
                                    block_size: int, num_heads: int, num_kv_heads: int,
                                    head_dim: int, scale: float, partition_blocks: int,
                                    workspace=None, workspace_bytes: int = 0,
                                    stream=None) -> None:
    _check(lib().pa_decode_attention_partitioned(
        _ptr(out), _ptr(q), pool, layer, _ptr(block_tables), max_blocks_per_seq,
        _ptr(context_lens), batch, block_size, num_heads, num_kv_heads, head_dim, float(scale),
        partition_blocks, _ptr(workspace), workspace_bytes, _stream(stream)),
        "pa_decode_attention_partitioned")


PA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def pa_decode_attention_noalloc(out, q, pool: int, layer: int, block_tables,
                                max_blocks_per_seq: int, context_lens, batch: int,
                                block_size: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                scale: float, partition_blocks: int = 0, stream=None) -> None:
    """Decode attention whose split-K scratch is the library's fixed device
    array (no device allocation by this call); see the header for its limits."""
    _check(lib().pa_decode_attention_noalloc(
        _ptr(out), _ptr(q), pool, layer, _ptr(block_tables), max_blocks_per_seq,
        _ptr(context_lens), batch, block_size, num_heads, num_kv_heads, head_dim, float(scale),
        partition_blocks, _stream(stream)), "pa_decode_attention_noalloc")


def pa_write_kv_and_decode(out, q, pool: int, layer: int, k, v, positions, block_tables,
                           max_blocks_per_seq: int, context_lens, batch: int, block_size: int,
                           num_heads: int, num_kv_heads: int, head_dim: int, scale: float,
                           partition_blocks: int = 0, workspace=None, workspace_bytes: int = 0,
                           stream=None) -> None:
    _check(lib().pa_write_kv_and_decode(
        _ptr(out), _ptr(q), pool, layer, _ptr(k), _ptr(v), _ptr(positions), _ptr(block_tables),
        max_blocks_per_seq, _ptr(context_lens), batch, block_size, num_heads, num_kv_heads,
        head_dim, float(scale), partition_blocks, _ptr(workspace), workspace_bytes,
        _stream(stream)), "pa_write_kv_and_decode")


def pa_gather_kv(k_out, v_out, mask, pool: int, layer: int, block_tables, max_blocks_per_seq: int,
                 context_lens, batch: int, max_len: int, stream=None) -> None:
    _check(lib().pa_gather_kv(_ptr(k_out), _ptr(v_out), _ptr(mask), pool, layer,
                              _ptr(block_tables), max_blocks_per_seq, _ptr(context_lens), batch,
                              max_len, _stream(stream)), "pa_gather_kv")


def pa_get_status(stream=None) -> int:
    v = ctypes.c_uint()
    _check(lib().pa_get_status(ctypes.byref(v), _stream(stream)), "pa_get_status")
    return v.value


def pa_selftest_wait_timeout(stream=None) -> None:
    _check(lib().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")
