"""``BlockPool``: a torch-owned pool tensor plus its library handle.

Mirrors the mini-infer BlockPool interface ("Paged KV-Cache Memory Management",
section "Python Implementation: Physical Block Pool": ``allocate_block``,
``free_block``, the [num_blocks, 2, num_layers, num_kv_heads, block_size,
head_dim] tensor) on top of the C ABI.  Marshalling only: torch allocates the
device memory, every operation runs in libpagedattn's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


_DECODE_KERNELS = {"auto": B.PA_DECODE_AUTO, "cuda_cores": B.PA_DECODE_CUDA_CORES,
                   "tensor_cores": B.PA_DECODE_TENSOR_CORES, "tcgen05": B.PA_DECODE_TCGEN05}


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int = 16, num_layers: int = 24,
                 num_kv_heads: int = 2, head_dim: int = 64, dtype=torch.bfloat16,
                 device="cuda", tensor: Optional[torch.Tensor] = None):
        shape = (num_blocks, 2, num_layers, num_kv_heads, block_size, head_dim)
        if tensor is None:
            tensor = torch.zeros(shape, dtype=dtype, device=device)
        if tuple(tensor.shape) != shape or not tensor.is_contiguous():
            raise ValueError(f"pool tensor must be contiguous with shape {shape}")
        self.pool = tensor
        self.num_blocks, self.block_size, self.num_layers = num_blocks, block_size, num_layers
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        self.dtype = tensor.dtype
        self.handle = B.pa_pool_create(tensor, num_blocks, num_layers, num_kv_heads, block_size,
                                       head_dim, tensor.dtype)

    # -- allocator ---------------------------------------------------------
    def allocate_block(self) -> int:
        return B.pa_alloc_block(self.handle)

    def free_block(self, block_id: int) -> None:
        B.pa_free_block(self.handle, block_id)

    def num_free(self) -> int:
        return B.pa_num_free(self.handle)

    def seed_free_stack(self, order) -> None:
        B.pa_pool_seed_free_stack(self.handle, order)

    def block_bytes(self) -> int:
        return B.pa_pool_block_bytes(self.handle)

    # -- the same free stack on the device (one launch per batch) -----------
    def device_stack(self, stream=None) -> torch.Tensor:
        """Moves the free stack into a new device tensor; the host allocator
        refuses until download_device_stack brings it back."""
        n = B.pa_device_stack_bytes(self.handle) // 4
        stack = torch.empty(n, dtype=torch.int32, device=self.pool.device)
        B.pa_device_stack_upload(self.handle, stack, stream)
        return stack

    def download_device_stack(self, stack: torch.Tensor, stream=None) -> None:
        B.pa_device_stack_download(self.handle, stack, stream)

    def device_allocate_blocks(self, stack: torch.Tensor, block_tables: torch.Tensor,
                               positions: torch.Tensor, stream=None) -> None:
        """Every sequence whose position starts a new block pops one from the
        device stack into its table (the order repeated host calls give)."""
        B.pa_device_alloc_blocks(self.handle, stack, block_tables, block_tables.shape[1],
                                 positions, positions.shape[0], stream)

    def device_allocate_blocks_step(self, stack: torch.Tensor, block_tables: torch.Tensor,
                                    positions: torch.Tensor, next_lens: torch.Tensor,
                                    stream=None) -> None:
        """device_allocate_blocks, and next_lens = positions + 1 in the same
        launch (the context lengths once this step's tokens are appended)."""
        B.pa_device_alloc_blocks_step(self.handle, stack, block_tables, block_tables.shape[1],
                                      positions, next_lens, positions.shape[0], stream)

    def device_free_blocks(self, stack: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, finished: torch.Tensor,
                           stream=None) -> None:
        """Finished sequences push their blocks back and their table rows become -1."""
        B.pa_device_free_blocks(self.handle, stack, block_tables, block_tables.shape[1],
                                context_lens, finished, context_lens.shape[0], stream)

    def set_decode_kernel(self, kind: str) -> None:
        """'auto' (default), 'cuda_cores', 'tensor_cores' (mma.sync) or 'tcgen05'."""
        B.pa_pool_set_decode_kernel(self.handle, _DECODE_KERNELS[kind])

    # -- kernels -----------------------------------------------------------
    def write_kv(self, layer: int, k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor,
                 positions: torch.Tensor, stream=None) -> None:
        B.pa_write_kv(self.handle, layer, k, v, block_tables, block_tables.shape[1], positions,
                      positions.shape[0], stream)

    def workspace_size(self, batch: int, num_heads: int, max_blocks_per_seq: int,
                       partition_blocks: int = 0) -> int:
        return B.pa_decode_workspace_size(self.handle, batch, num_heads, max_blocks_per_seq,
                                          partition_blocks)

    def decode_attention(self, q: torch.Tensor, layer: int, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, scale: float,
                         out: Optional[torch.Tensor] = None, partition_blocks: int = 0,
                         workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        batch, num_heads, head_dim = q.shape
        maxb = block_tables.shape[1]
        if out is None:
            out = torch.empty((batch, num_heads, head_dim), dtype=torch.float32, device=q.device)
        need = self.workspace_size(batch, num_heads, maxb, partition_blocks)
        if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        B.pa_decode_attention_partitioned(out, q, self.handle, layer, block_tables, maxb,
                                          context_lens, batch, self.block_size, num_heads,
                                          self.num_kv_heads, head_dim, scale, partition_blocks,
                                          workspace, wbytes, stream)
        return out

    def write_kv_and_decode(self, q: torch.Tensor, layer: int, k: torch.Tensor, v: torch.Tensor,
                            positions: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, scale: float,
                            out: Optional[torch.Tensor] = None, partition_blocks: int = 0,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """write_kv then decode_attention in one launch (context_lens normally
        include the new token)."""
        batch, num_heads, head_dim = q.shape
        maxb = block_tables.shape[1]
        if out is None:
            out = torch.empty((batch, num_heads, head_dim), dtype=torch.float32, device=q.device)
        need = self.workspace_size(batch, num_heads, maxb, partition_blocks)
        if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        B.pa_write_kv_and_decode(out, q, self.handle, layer, k, v, positions, block_tables, maxb,
                                 context_lens, batch, self.block_size, num_heads,
                                 self.num_kv_heads, head_dim, scale, partition_blocks, workspace,
                                 wbytes, stream)
        return out

    def gather_kv(self, layer: int, block_tables: torch.Tensor, context_lens: torch.Tensor,
                  max_len: int, stream=None):
        batch = context_lens.shape[0]
        shape = (batch, max_len, self.num_kv_heads, self.head_dim)
        k = torch.empty(shape, dtype=self.dtype, device=self.pool.device)
        v = torch.empty(shape, dtype=self.dtype, device=self.pool.device)
        mask = torch.empty((batch, max_len), dtype=torch.uint8, device=self.pool.device)
        B.pa_gather_kv(k, v, mask, self.handle, layer, block_tables, block_tables.shape[1],
                       context_lens, batch, max_len, stream)
        return k, v, mask.bool()

    def close(self) -> None:
        if getattr(self, "handle", None):
            B.pa_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
