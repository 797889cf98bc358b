"""A decode step over the C ABI: owner-filtered append -> partials -> merge.

``ShardedMlaDecoder`` owns the device buffers of one sharded MLA layer held on
this GPU (the pools of shards [shard_begin, shard_end), the partial outputs,
the merged output and the library workspace), all allocated once through
PyTorch.  Each method is a fixed sequence of C-ABI calls; no arithmetic of the
method happens here.

The library's host work per call depends only on shapes, pointers and the
device (every length is read on the device), and nothing here synchronises or
allocates per call, so a whole ``step`` can be captured once in a CUDA graph
(``torch.cuda.graph``) and replayed with new lengths, queries and rows written
in place into the captured tensors.
"""

from __future__ import annotations

import torch

from . import (DCP_LSE_BASE_2, DCP_LSE_BASE_E, Layout, dcp_kv_append, dcp_lse_merge,
               dcp_mla_decode_partial, dcp_mla_decode_workspace_size)


class ShardedMlaDecoder:
    def __init__(self, layout: Layout, B: int, q_len: int, H: int, pool_pages: int, max_pages: int,
                 scale: float, lse_base: int = DCP_LSE_BASE_E, out_dtype=torch.bfloat16,
                 part_dtype=torch.float32, shard_begin: int = 0, shard_end: int | None = None,
                 device="cuda"):
        self.layout = layout
        self.shard_begin = shard_begin
        self.shard_end = layout.n_shards if shard_end is None else shard_end
        n = self.shard_end - self.shard_begin
        self.B, self.q_len, self.H = B, q_len, H
        self.pool_pages, self.max_pages = pool_pages, max_pages
        self.scale = scale
        self.lse_base = lse_base
        dev = torch.device(device)
        self.arena = torch.zeros(n, pool_pages * layout.page_size, 576, dtype=torch.bfloat16, device=dev)
        self.o_part = torch.empty(n, B, q_len, H, 512, dtype=part_dtype, device=dev)
        self.lse_part = torch.empty(n, B, q_len, H, dtype=torch.float32, device=dev)
        self.o = torch.empty(B, q_len, H, 512, dtype=out_dtype, device=dev)
        self.lse = torch.empty(B, q_len, H, dtype=torch.float32, device=dev)
        ws = dcp_mla_decode_workspace_size(layout, self.shard_begin, self.shard_end, B, q_len, H)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def append(self, kv_new, pos, req, block_table, stream=None):
        """Place T new latent rows (kv_new [T, 576] bf16 at positions pos of requests req):
        one owner-filtered append, placement computed in the kernel."""
        if kv_new.shape[0] == 0:
            return
        dcp_kv_append(self.layout, self.shard_begin, self.shard_end, kv_new, pos, req, block_table,
                      self.max_pages, self.arena, self.pool_pages, self.status, stream)

    def partial(self, q, block_table, seq_lens, stream=None):
        dcp_mla_decode_partial(self.layout, self.shard_begin, self.shard_end, q, self.arena,
                               self.pool_pages, block_table, self.max_pages, seq_lens, self.scale,
                               self.lse_base, self.o_part, self.lse_part, self.workspace, self.status,
                               stream)

    def merge(self, stream=None):
        n = self.shard_end - self.shard_begin
        dcp_lse_merge(self.o_part.view(n, -1, 512), self.lse_part.view(n, -1), self.lse_base,
                      self.o.view(-1, 512), self.lse.view(-1), stream)

    def decode(self, q, block_table, seq_lens, stream=None):
        """Partials of every held shard, then their merge into self.o / self.lse."""
        self.partial(q, block_table, seq_lens, stream)
        self.merge(stream)
        return self.o, self.lse

    def step(self, q, block_table, seq_lens, kv_new=None, pos=None, req=None, stream=None):
        """One decode step: append this step's tokens (if any), then decode."""
        if kv_new is not None:
            self.append(kv_new, pos, req, block_table, stream)
        return self.decode(q, block_table, seq_lens, stream)

    def status_bits(self) -> int:
        return int(self.status.item())


__all__ = ["ShardedMlaDecoder", "DCP_LSE_BASE_E", "DCP_LSE_BASE_2"]
