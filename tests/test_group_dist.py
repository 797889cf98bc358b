"""The multi-GPU exchange's host logic over gloo on CPU (world sizes 2 and 4).

Each process is one rank of a DCP group.  It drives the library's own
``DcpExchange`` (buffer layout, shard and head ranges, the all-to-all /
all-gather / reduce-scatter calls) with the kernels replaced by the oracle's
restatement of them (wire-format pack, packed merge, local rescale), so that
the collective path runs without a GPU.  Checks, on every rank d:
  * the receive buffer holds exactly head slice d of every shard, in shard
    order, bit for bit what a one-process layout of all ranks' sends gives;
  * the merged output of d's heads equals the oracle's strategy end to end and
    unsharded attention.
The CUDA kernels themselves are checked against the same oracle on the GPU
(tests/test_gpu_group.py).
"""

import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import attention, exchange

SCALE = 1.0 / math.sqrt(192.0)


class OracleOps:
    """The exchange kernels' contracts, computed by the oracle on CPU tensors."""

    def __init__(self, T, H, base):
        self.T, self.H, self.base = T, H, base

    @staticmethod
    def dcp_a2a_chunk_bytes(n_held, T, H, world, wire_dtype=torch.bfloat16):
        return exchange.chunk_bytes(n_held, T, H, world, wire_dtype == torch.bfloat16)

    @staticmethod
    def dcp_pack_partials(o_part, lse_part, world, send, wire_dtype=torch.bfloat16, stream=None):
        n = o_part.shape[0]
        H = o_part.shape[-2]
        buf = exchange.pack(o_part.double().numpy().reshape(n, -1, H, 512), lse_part.double().numpy().reshape(n, -1, H),
                            world, wire_dtype == torch.bfloat16)
        send.copy_(torch.from_numpy(buf))

    def dcp_lse_merge_packed(self, recv, world, n_held, lse_base, o, lse=None, wire_dtype=torch.bfloat16,
                             stream=None):
        o_, l_ = exchange.merge_received(recv.numpy(), n_held, self.T, self.H, world, wire_dtype == torch.bfloat16,
                                         lse_base)
        o.copy_(torch.from_numpy(o_).reshape(o.shape))
        if lse is not None:
            lse.copy_(torch.from_numpy(l_).reshape(lse.shape))

    @staticmethod
    def dcp_lse_rescale(lse_all, o_part, shard_begin, world, lse_base, o_sum, lse=None, stream=None):
        o_, l_ = exchange.rescale_local(lse_all.double().numpy(), o_part.double().numpy(), shard_begin, world,
                                        lse_base)
        o_sum.copy_(torch.from_numpy(o_).reshape(o_sum.shape))
        if lse is not None:
            lse.copy_(torch.from_numpy(l_).reshape(lse.shape))


def case(N, T, H, base, seed=7):
    """Every shard's partials of one request with T query tokens (q_len = T, causal)."""
    rng = np.random.default_rng(seed)
    S = 3 * N + 5
    q = rng.standard_normal((T, H, 576))
    kv = rng.standard_normal((S, 576))
    _o, _l, o_p, l_p = attention.sharded_attention(q, kv, S, N, 1, SCALE, base)
    o_ref, l_ref = attention.attention(q, kv, S, SCALE, base)
    return o_p, l_p, o_ref, l_ref


def _rank_main(rank, world, port, N, T, H, base, strategy, wire_bf16):
    import torch.distributed as dist
    from context_sharded_mla_gb300.group import DcpExchange
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        o_p, l_p, o_ref, l_ref = case(N, T, H, base)
        wire = torch.bfloat16 if wire_bf16 else torch.float32
        x = DcpExchange(world, rank, N, T, H, base, strategy, wire, torch.float32, "cpu",
                        ops=OracleOps(T, H, base), dist=dist)
        s0, s1 = x.shard_begin, x.shard_end
        assert (s0, s1) == exchange.shard_range(rank, N, world)
        o_held = torch.from_numpy(o_p[s0:s1]).float()
        l_held = torch.from_numpy(l_p[s0:s1]).float()
        o, lse = x.exchange(o_held, l_held)
        h0, h1 = exchange.head_range(rank, H, world)
        assert (h0, h1) == (x.head_begin, x.head_end)
        if strategy == "a2a":
            # what a one-process layout of every rank's send buffer hands to rank `rank`
            n = N // world
            want = np.stack([exchange.pack(o_p[w * n:(w + 1) * n].astype(np.float32),
                                           l_p[w * n:(w + 1) * n].astype(np.float32), world, wire_bf16)[rank]
                             for w in range(world)])
            assert np.array_equal(x.recv.numpy(), want), f"rank {rank}: receive buffer differs"
            ref = exchange.a2a_merge(o_p.astype(np.float32).astype(np.float64),
                                     l_p.astype(np.float32).astype(np.float64), world, base)[rank]
        else:
            ref = exchange.ag_rs_merge(o_p.astype(np.float32).astype(np.float64),
                                       l_p.astype(np.float32).astype(np.float64), world, base)[rank]
        # bf16 on the wire: the output tolerance of the decode path, |err| <= 1e-2 + 1e-2 |ref|
        tol = 1e-2 if wire_bf16 else 1e-5
        assert np.allclose(o.double().numpy(), ref[0], rtol=tol, atol=tol), f"rank {rank}: o"
        assert np.allclose(lse.double().numpy(), ref[1], rtol=1e-5, atol=1e-5), f"rank {rank}: lse"
        assert np.allclose(o.double().numpy(), o_ref[:, h0:h1], rtol=tol, atol=tol)
        assert np.allclose(lse.double().numpy(), l_ref[:, h0:h1], rtol=1e-5, atol=1e-5)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,N,T,H,base,strategy,wire_bf16", [
    (2, 8, 3, 8, 2, "a2a", True),
    (2, 2, 1, 4, 0, "a2a", False),
    (4, 8, 2, 8, 0, "a2a", True),
    (2, 8, 3, 8, 2, "ag_rs", False),
    (4, 16, 2, 8, 0, "ag_rs", False),
])
def test_exchange_over_gloo(world, N, T, H, base, strategy, wire_bf16):
    mp.spawn(_rank_main, args=(world, _free_port(), N, T, H, base, strategy, wire_bf16), nprocs=world, join=True)


def test_ranges_reject_uneven_splits():
    from context_sharded_mla_gb300.group import head_range, shard_range
    assert shard_range(3, 8, 4) == (6, 8) and head_range(1, 96, 8) == (12, 24)
    with pytest.raises(ValueError):
        shard_range(0, 8, 3)
    with pytest.raises(ValueError):
        head_range(0, 96, 7)
