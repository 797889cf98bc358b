"""The multi-GPU decode path's kernels on one GPU, against the fp64 oracle.

W ranks are emulated in one process: each rank is a DcpGroupDecoder with its
own shard range and pools (the append filters by owner), and runs the real
kernels: partials of its shards for all heads, then dcp_pack_partials +
dcp_lse_merge_packed (all-to-all form) or dcp_lse_rescale (AllGather +
ReduceScatter form).  The collectives between the phases are plain device
copies (the all-to-all moves chunk d of rank w's send buffer to chunk w of rank
d's receive buffer; the reduce-scatter sums the ranks' blocks), so no kernel
waits on another rank.  Each rank's merged heads are compared with the oracle's
unsharded attention of those heads.  The world-size-1 path of the decoder runs
as the library runs it (no collective).  A property check pins the pack's byte
layout on the full-size K3 partials: each chunk is a head slice of o_part.
"""

import pytest
import torch

import workloads
from oracle import attention

from harness import assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu


def _ranks(cfg, world, strategy, wire, out_dtype):
    import context_sharded_mla_gb300 as dcp
    from context_sharded_mla_gb300.group import DcpGroupDecoder
    dcp.load_library()
    dev = torch.device("cuda")
    S = workloads.lengths(cfg)
    bt, pool_pages = workloads.block_table(cfg, S)
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    ranks = [DcpGroupDecoder(lay, cfg.B, cfg.q_len, cfg.H, pool_pages, bt.shape[1], workloads.SCALE, w, world,
                             1 if cfg.base == 2 else 0, strategy, wire, out_dtype, device=dev)
             for w in range(world)]
    btd = bt.to(dev)
    kvs = []
    for b in range(cfg.B):
        kv = workloads.gen_kv(cfg, b, int(S[b]))
        kvs.append(kv)
        pos = torch.arange(int(S[b]), device=dev)
        req = torch.full((int(S[b]),), b, dtype=torch.int32, device=dev)
        for r in ranks:                                   # every rank sees every token, keeps its own
            r.append(kv.to(dev), pos, req, btd)
    q = workloads.gen_q(cfg)
    return ranks, q, kvs, S, btd


def _oracle(cfg, q, kvs, S):
    return [attention.attention(to_f64(q[b]), to_f64(kvs[b]), int(S[b]), workloads.SCALE, cfg.base)
            for b in range(cfg.B)]


def _check_rank(cfg, r, o, lse, ref):
    h0, h1 = r.head_begin, r.head_end
    o = to_f64(o).reshape(cfg.B, cfg.q_len, h1 - h0, 512)
    lse = to_f64(lse).reshape(cfg.B, cfg.q_len, h1 - h0)
    for b in range(cfg.B):
        assert_close_o(o[b], ref[b][0][:, h0:h1], f"rank heads [{h0},{h1}) b={b}")
        assert_close_lse(lse[b], ref[b][1][:, h0:h1], f"rank heads [{h0},{h1}) b={b}")


@pytest.mark.parametrize("name,over,world,strategy,wire", [
    ("k3", dict(B=3, S=4096 + 13), 8, "a2a", torch.bfloat16),     # one shard per rank, base 2
    ("k3", dict(B=2, S=3000), 2, "a2a", torch.float32),           # four shards per rank, f32 wire
    ("dsv3", dict(B=2, S=2 * 8 * 128 + 37), 4, "ag_rs", None),
    ("ragged", dict(B=3, S=3000, S_min=17), 4, "a2a", torch.bfloat16),   # I = 16, causal q_len 4
    ("ragged", dict(B=2, S=2000, S_min=300), 16, "ag_rs", None),
    ("extend", dict(B=2, S=3000 + 5, H=32), 2, "a2a", torch.bfloat16),   # 64 causal query tokens
])
def test_emulated_group_matches_oracle(name, over, world, strategy, wire):
    import context_sharded_mla_gb300 as dcp
    cfg = workloads.config(name, **over)
    out_dtype = torch.float32 if strategy == "ag_rs" else torch.bfloat16
    ranks, q, kvs, S, btd = _ranks(cfg, world, strategy, wire or torch.bfloat16, out_dtype)
    qd = q.to("cuda")
    seq = S.to("cuda")
    for r in ranks:                                       # phase 1: partials (and pack) on every rank
        r.local.partial(qd, btd, seq)
        if strategy == "a2a":
            dcp.dcp_pack_partials(r.local.o_part, r.local.lse_part, world, r.xchg.send, wire)
    if strategy == "a2a":                                 # phase 2: the all-to-all, as device copies
        for d, rd in enumerate(ranks):
            for w, rw in enumerate(ranks):
                rd.xchg.recv[w].copy_(rw.xchg.send[d])
        for r in ranks:                                   # phase 3: each head owner merges
            x = r.xchg
            dcp.dcp_lse_merge_packed(x.recv, world, x.n_held, x.lse_base, x.o.view(-1, 512), x.lse.view(-1), wire)
    else:
        lse_all = torch.cat([r.local.lse_part for r in ranks]).view(cfg.N, -1, cfg.H)
        for r in ranks:
            x = r.xchg
            dcp.dcp_lse_rescale(lse_all, r.local.o_part, x.shard_begin, world, x.lse_base, x.o_sum, x.lse_blocks)
        for d, rd in enumerate(ranks):                    # the reduce-scatter: rank d sums block d
            rd.xchg.o.copy_(torch.stack([rw.xchg.o_sum[d] for rw in ranks]).sum(0))
    torch.cuda.synchronize()
    ref = _oracle(cfg, q, kvs, S)
    for r in ranks:
        assert r.status_bits() == 0
        _check_rank(cfg, r, r.xchg.o, r.xchg.lse, ref)


@pytest.mark.parametrize("strategy", ["a2a", "ag_rs"])
def test_world_size_one_decoder(strategy):
    cfg = workloads.config("k3", B=3, S=5000)
    ranks, q, kvs, S, btd = _ranks(cfg, 1, strategy, torch.bfloat16, torch.bfloat16)
    o, lse = ranks[0].decode(q.to("cuda"), btd, S.to("cuda"))
    torch.cuda.synchronize()
    assert ranks[0].status_bits() == 0
    _check_rank(cfg, ranks[0], o, lse, _oracle(cfg, q, kvs, S))


@pytest.mark.parametrize("part_dtype,wire", [(torch.float32, torch.bfloat16), (torch.bfloat16, torch.bfloat16),
                                             (torch.float32, torch.float32)])
def test_pack_chunks_are_head_slices(part_dtype, wire):
    """Property at any size: chunk d of the send buffer is head slice d of o_part (in the
    wire dtype, rounded to nearest even) followed by the same slice of lse_part."""
    import context_sharded_mla_gb300 as dcp
    dcp.load_library()
    g = torch.Generator(device="cuda").manual_seed(5)
    n_held, T, H, world = 1, 64, 96, 8                    # the K3 step on 8 ranks
    o_part = torch.randn(n_held, T, H, 512, generator=g, device="cuda").to(part_dtype)
    lse_part = torch.randn(n_held, T, H, generator=g, device="cuda")
    lse_part[0, 3, 5] = float("-inf")
    chunk = dcp.dcp_a2a_chunk_bytes(n_held, T, H, world, wire)
    send = torch.zeros(world, chunk, dtype=torch.uint8, device="cuda")
    dcp.dcp_pack_partials(o_part, lse_part, world, send, wire)
    torch.cuda.synchronize()
    Hd = H // world
    e = 2 if wire == torch.bfloat16 else 4
    ob = n_held * T * Hd * 512 * e
    for d in range(world):
        o_blk = send[d, :ob].view(wire).view(n_held, T, Hd, 512)
        l_blk = send[d, ob:ob + n_held * T * Hd * 4].view(torch.float32).view(n_held, T, Hd)
        assert torch.equal(o_blk, o_part[:, :, d * Hd:(d + 1) * Hd].to(wire))
        assert torch.equal(l_blk, lse_part[:, :, d * Hd:(d + 1) * Hd])
