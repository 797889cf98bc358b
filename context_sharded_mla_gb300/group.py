"""Decode Context Parallelism across GPUs: one rank per GPU, N / W shards each.

Rank w of a W-rank group holds the context shards [w*N/W, (w+1)*N/W) of every
request and owns the heads [w*H/W, (w+1)*H/W) of the output.  A decode step on
a rank is: owner-filtered append of the new tokens (its shards only), the
partials of its shards for ALL heads (the query is replicated on every rank,
the pages' "copy the projection" option), then the exchange that hands each
head owner the partials of its heads from every shard, and their merge.

Two exchange strategies ("Decode Context Parallelism" (zdszero), "通信策略"):

* ``"a2a"`` (default): pack each rank's partials by head slice, o and lse in
  one buffer (dcp_pack_partials), one all-to-all, and the head owner's LSE
  merge read in place from the receive buffer (dcp_lse_merge_packed).  One
  collective per layer ("MLA 的 Decode Context Parallelism", section 4, stages
  6-7).
* ``"ag_rs"``: all-gather every shard's lse, correct this rank's partials to
  exp(lse_r - L) o_r summed over its shards (dcp_lse_rescale), and a
  reduce-scatter (sum) by head.  Two collectives; the output is f32.

Every step of the arithmetic runs in the library's CUDA kernels; this module
only holds buffers and issues the calls and the collectives
(``torch.distributed``, NCCL on GPUs).  ``DcpExchange`` takes the kernel
functions as ``ops`` (the CUDA binding by default), so that its host logic, the
buffer layout and the collective calls, can also be driven with CPU tensors
over gloo.
"""

from __future__ import annotations

import torch

from . import DCP_LSE_BASE_E, Layout
from .step import ShardedMlaDecoder


def shard_range(rank: int, n_shards: int, world: int):
    """Shards [begin, end) held by `rank` (n_shards % world == 0)."""
    if world < 1 or n_shards % world:
        raise ValueError(f"{n_shards} shards do not split evenly over {world} ranks")
    n = n_shards // world
    return rank * n, (rank + 1) * n


def head_range(rank: int, H: int, world: int):
    """Heads [begin, end) owned by `rank` after the exchange (H % world == 0)."""
    if world < 1 or H % world:
        raise ValueError(f"{H} heads do not split evenly over {world} ranks")
    n = H // world
    return rank * n, (rank + 1) * n


def _cuda_ops():
    from . import dcp_a2a_chunk_bytes, dcp_lse_merge_packed, dcp_lse_rescale, dcp_pack_partials

    class _Ops:
        pass
    ops = _Ops()
    ops.dcp_a2a_chunk_bytes = dcp_a2a_chunk_bytes
    ops.dcp_pack_partials = dcp_pack_partials
    ops.dcp_lse_merge_packed = dcp_lse_merge_packed
    ops.dcp_lse_rescale = dcp_lse_rescale
    return ops


class DcpExchange:
    """The exchange of one rank's partials (o_part [n_held, T, H, 512], lse_part
    [n_held, T, H]) with the head owners; buffers are allocated once."""

    def __init__(self, world: int, rank: int, n_shards: int, T: int, H: int, lse_base: int = DCP_LSE_BASE_E,
                 strategy: str = "a2a", wire_dtype=torch.bfloat16, out_dtype=torch.bfloat16, device="cuda",
                 group=None, ops=None, dist=None):
        if strategy not in ("a2a", "ag_rs"):
            raise ValueError(f"unknown exchange strategy {strategy!r}")
        self.world, self.rank, self.n_shards, self.T, self.H = world, rank, n_shards, T, H
        self.shard_begin, self.shard_end = shard_range(rank, n_shards, world)
        self.head_begin, self.head_end = head_range(rank, H, world)
        self.n_held = self.shard_end - self.shard_begin
        self.Hd = H // world
        self.lse_base = lse_base
        self.strategy = strategy
        self.wire_dtype = wire_dtype
        self.group = group
        self.ops = ops if ops is not None else _cuda_ops()
        if dist is None and world > 1:
            import torch.distributed as dist
        self.dist = dist
        dev = torch.device(device)
        if strategy == "a2a":
            self.chunk = self.ops.dcp_a2a_chunk_bytes(self.n_held, T, H, world, wire_dtype)
            self.send = torch.empty(world, self.chunk, dtype=torch.uint8, device=dev)
            self.recv = torch.empty_like(self.send) if world > 1 else self.send
            self.o = torch.empty(T, self.Hd, 512, dtype=out_dtype, device=dev)
            self.lse = torch.empty(T, self.Hd, dtype=torch.float32, device=dev)
        else:
            self.lse_all = torch.empty(n_shards, T, H, dtype=torch.float32, device=dev) if world > 1 else None
            self.o_sum = torch.empty(world, T, self.Hd, 512, dtype=torch.float32, device=dev)
            self.lse_blocks = torch.empty(world, T, self.Hd, dtype=torch.float32, device=dev)
            self.o = torch.empty(T, self.Hd, 512, dtype=torch.float32, device=dev) if world > 1 else self.o_sum[0]
            self.lse = self.lse_blocks[rank]

    def bytes_sent(self) -> int:
        """Bytes this rank hands to the collectives per step (its own chunk included)."""
        if self.strategy == "a2a":
            return self.send.numel()
        return self.n_held * self.T * self.H * 4 + self.o_sum.numel() * 4

    def exchange(self, o_part, lse_part, stream=None):
        """(o [T, Hd, 512], lse [T, Hd]) of this rank's heads, merged over every shard.

        Kernels and collectives are ordered on one stream: `stream` if given (it
        becomes the current stream for the call), else the current stream."""
        if stream is not None:
            with torch.cuda.stream(stream):
                return self._exchange(o_part, lse_part)
        return self._exchange(o_part, lse_part)

    def _exchange(self, o_part, lse_part):
        ops = self.ops
        if self.strategy == "a2a":
            ops.dcp_pack_partials(o_part, lse_part, self.world, self.send, self.wire_dtype)
            if self.world > 1:
                self.dist.all_to_all_single(self.recv.view(-1), self.send.view(-1), group=self.group)
            ops.dcp_lse_merge_packed(self.recv, self.world, self.n_held, self.lse_base, self.o.view(-1, 512),
                                     self.lse.view(-1), self.wire_dtype)
            return self.o, self.lse
        if self.world > 1:
            self.dist.all_gather_into_tensor(self.lse_all.view(-1), lse_part.reshape(-1), group=self.group)
            lse_all = self.lse_all
        else:
            lse_all = lse_part.reshape(self.n_shards, self.T, self.H)
        ops.dcp_lse_rescale(lse_all, o_part, self.shard_begin, self.world, self.lse_base, self.o_sum,
                            self.lse_blocks)
        if self.world > 1:
            self.dist.reduce_scatter_tensor(self.o.view(-1), self.o_sum.view(-1), group=self.group)
        return self.o, self.lse


class DcpGroupDecoder:
    """One rank's decode step: its shards' pools, partials and the exchange."""

    def __init__(self, layout: Layout, B: int, q_len: int, H: int, pool_pages: int, max_pages: int, scale: float,
                 rank: int, world: int, lse_base: int = DCP_LSE_BASE_E, strategy: str = "a2a",
                 wire_dtype=torch.bfloat16, out_dtype=torch.bfloat16, part_dtype=torch.float32, group=None,
                 device="cuda"):
        sb, se = shard_range(rank, layout.n_shards, world)
        self.B, self.q_len, self.H = B, q_len, H
        self.local = ShardedMlaDecoder(layout, B, q_len, H, pool_pages, max_pages, scale, lse_base, out_dtype,
                                       part_dtype, shard_begin=sb, shard_end=se, device=device)
        self.xchg = DcpExchange(world, rank, layout.n_shards, B * q_len, H, lse_base, strategy, wire_dtype,
                                out_dtype, device, group)
        self.head_begin, self.head_end = self.xchg.head_begin, self.xchg.head_end

    @property
    def status(self):
        return self.local.status

    def append(self, kv_new, pos, req, block_table, stream=None):
        self.local.append(kv_new, pos, req, block_table, stream)

    def decode(self, q, block_table, seq_lens, stream=None):
        """Partials of this rank's shards for all heads, then the exchange: returns
        (o [B, q_len, H/W, 512], lse [B, q_len, H/W]) of this rank's heads."""
        if stream is not None:
            with torch.cuda.stream(stream):
                return self.decode(q, block_table, seq_lens)
        self.local.partial(q, block_table, seq_lens)
        o, lse = self.xchg.exchange(self.local.o_part, self.local.lse_part)
        Hd = self.head_end - self.head_begin
        return o.view(self.B, self.q_len, Hd, 512), lse.view(self.B, self.q_len, Hd)

    def step(self, q, block_table, seq_lens, kv_new=None, pos=None, req=None, stream=None):
        if kv_new is not None:
            self.append(kv_new, pos, req, block_table, stream)
        return self.decode(q, block_table, seq_lens, stream)

    def status_bits(self) -> int:
        return self.local.status_bits()


__all__ = ["DcpExchange", "DcpGroupDecoder", "shard_range", "head_range"]
