"""GPU parity of the decode partial and the LSE merge against the fp64 oracle.

Sizes are small enough for the oracle to finish in seconds but span several
KV tiles per shard and a ragged tail; every workload family is covered
(token RR and interleave 16, base e and base 2, q_len 1, causal q_len 4 and
the 64-token chunked extend, fp32 and bf16 partials), plus empty shards,
needles and the merge alone.
Tolerance (written here, from the stated bar): |err| <= 1e-2 + 1e-2 |ref| for
outputs, 1e-3 absolute for lse.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention

from harness import GpuState, assert_close_lse, assert_close_o, rel_row_err, to_f64

pytestmark = pytest.mark.gpu


def _check_state(st, reqs=None, heads=None, check_parts=True, rel_bound=None):
    o, lse = st.decode()
    cfg = st.cfg
    o = to_f64(o)
    lse = to_f64(lse)
    o_part = to_f64(st.dec.o_part)
    lse_part = to_f64(st.dec.lse_part)
    reqs = range(cfg.B) if reqs is None else reqs
    worst = 0.0
    for b in reqs:
        ref_o, ref_lse, ref_op, ref_lp = st.oracle_request(b, heads)
        hs = slice(None) if heads is None else heads
        assert_close_o(o[b][:, hs], ref_o, f"merged o b={b}")
        assert_close_lse(lse[b][:, hs], ref_lse, f"merged lse b={b}")
        worst = max(worst, rel_row_err(o[b][:, hs], ref_o))
        if check_parts:
            for r in range(cfg.N):
                assert_close_o(o_part[r, b][:, hs], ref_op[r], f"o_part r={r} b={b}")
                assert_close_lse(lse_part[r, b][:, hs], ref_lp[r], f"lse_part r={r} b={b}")
    if rel_bound is not None:
        assert worst <= rel_bound, f"row-relative error {worst:.3e} > {rel_bound}"
    assert st.dec.status_bits() == 0
    return worst


SMALL = {
    "tiny": dict(),
    "dsv3": dict(B=2, S=2 * 8 * 128 + 37),
    "k3": dict(B=3, S=4096 + 13),
    "ragged": dict(B=5, S=3000, S_min=17),
    "long": dict(B=2, S=20000 + 7),
    "extend": dict(B=2, S=3000 + 5, H=32),   # 64 causal query tokens x 32 heads = 16 row groups
}


@pytest.mark.parametrize("name", list(SMALL))
def test_partial_and_merge_small(name):
    cfg = workloads.config(name, **SMALL[name])
    st = GpuState(cfg)
    _check_state(st, rel_bound=2e-2)


@pytest.mark.parametrize("name", ["k3", "dsv3", "ragged"])
def test_needle_small(name):
    """A planted needle makes one token (one shard) dominate: o is O(1)."""
    cfg = workloads.config(name, **SMALL[name])
    st = GpuState(cfg, needle=True)
    worst = _check_state(st, rel_bound=2e-2)
    o = to_f64(st.dec.o)
    for b in range(cfg.B):
        h = b % cfg.H
        ref = to_f64(st.kv[b][int(st.needle_pos[b])])[:512]
        # the needle head's output is (almost) the needle row itself
        assert np.max(np.abs(o[b, 0, h] - ref)) < 5e-2 + 2e-2 * np.max(np.abs(ref))
    # plain averaging of the partials is visibly wrong on these rows
    o_part = to_f64(st.dec.o_part)
    b, h = 0, 0
    avg = o_part[:, b, 0, h].mean(axis=0)
    assert np.max(np.abs(avg - o[b, 0, h])) > 0.1


@pytest.mark.parametrize("H,N", [(96, 8), (128, 8), (16, 4)])
def test_running_max_jumps(H, N):
    """Rows whose running maximum jumps several times inside one shard's stream.

    Three planted rows (query copies scaled 0.5, 1.0, 1.5: scores ~20, 40, 60)
    sit late in the sequence, so the kernel must rescale accumulated outputs
    in the middle of a work range, with many tiles per CTA.
    """
    import context_sharded_mla_gb300 as dcp
    from context_sharded_mla_gb300.step import ShardedMlaDecoder
    S_total = 40000 + 33
    cfg = workloads.config("k3", B=2, H=H, N=N, S=S_total)
    S = workloads.lengths(cfg)
    bt, pool_pages = workloads.block_table(cfg, S)
    dev = "cuda"
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    dec = ShardedMlaDecoder(lay, cfg.B, 1, cfg.H, pool_pages, bt.shape[1], workloads.SCALE, 1)
    q = workloads.gen_q(cfg)
    btd = bt.to(dev)
    kvs = []
    for b in range(cfg.B):
        kv = workloads.gen_kv(cfg, b, int(S[b]))
        for f, p in zip((0.5, 1.0, 1.5), (S_total // 2 + 7, 3 * S_total // 4 + 1, S_total - 100)):
            kv[p] = (q[b, 0, b % H].float() * f).to(torch.bfloat16)
        kvs.append(kv)
        n = int(S[b])
        dec.append(kv.to(dev), torch.arange(n, device=dev), torch.full((n,), b, dtype=torch.int32, device=dev), btd)
    o, lse = dec.decode(q.to(dev), btd, S.to(dev))
    torch.cuda.synchronize()
    assert dec.status_bits() == 0
    for b in range(cfg.B):
        ro, rl, rop, rlp = attention.sharded_attention(to_f64(q[b]), to_f64(kvs[b]), int(S[b]), cfg.N, cfg.I,
                                                       workloads.SCALE, 2)
        assert_close_o(to_f64(o[b]), ro, "jump o")
        assert_close_lse(to_f64(lse[b]), rl, "jump lse")
        for r in range(cfg.N):
            assert_close_o(to_f64(dec.o_part[r, b]), rop[r], f"jump o_part r={r}")
            assert_close_lse(to_f64(dec.lse_part[r, b]), rlp[r], f"jump lse_part r={r}")


@pytest.mark.parametrize("name,over", [
    ("k3", SMALL["k3"]),                                    # 96 rows: every softmax warp full
    ("k3", dict(B=3, S=3000 + 9, H=40)),                    # 40 rows in a 48-row group: a warp with 8 rows
    ("ragged", dict(B=4, S=2500, S_min=40, H=5)),           # 20 rows (q_len 4 x 5 heads): a warp with 4 rows
])
@pytest.mark.parametrize("part_dtype", [torch.bfloat16, torch.float32])
def test_partial_rows_of_both_dtypes(name, over, part_dtype):
    """The epilogue writes each warp's rows through shared memory; groups whose
    last warp has fewer than 16 rows must write only those rows."""
    cfg = workloads.config(name, **over)
    st = GpuState(cfg, part_dtype=part_dtype)
    _check_state(st, rel_bound=2e-2 if part_dtype == torch.bfloat16 else None)


@pytest.mark.parametrize("N,I,P,q_len", [(16, 16, 64, 4), (8, 1, 64, 1), (4, 2, 16, 4)])
def test_edge_lengths_empty_shards(N, I, P, q_len):
    """Lengths 1 .. N*I+1: many shards are empty (lse = -inf, o = 0) and rows see few tokens."""
    cfg0 = workloads.config("ragged", B=N * I + 1, N=N, I=I, P=P, q_len=q_len, H=8)
    cfg = workloads.config("ragged", B=N * I + 1, N=N, I=I, P=P, q_len=q_len, H=8,
                           lengths_override=workloads.edge_lengths(cfg0))
    st = GpuState(cfg)
    _check_state(st)
    lse_part = to_f64(st.dec.lse_part)
    assert np.isneginf(lse_part).any()           # some shards really are empty
    o_part = to_f64(st.dec.o_part)
    assert np.all(o_part[np.isneginf(lse_part)] == 0.0)


def test_base2_matches_base_e():
    cfg = workloads.config("k3", **SMALL["k3"])
    st2 = GpuState(cfg)
    o2, lse2 = [to_f64(t) for t in st2.decode()]
    cfg_e = workloads.config("k3", base=0, **SMALL["k3"])
    ste = GpuState(cfg_e)
    oe, lsee = [to_f64(t) for t in ste.decode()]
    assert np.allclose(lse2, lsee * math.log2(math.e), atol=1e-3)
    assert_close_o(o2, oe, "base-2 vs base-e output")


@pytest.mark.parametrize("in_dtype,out_dtype,base", [
    (torch.float32, torch.float32, 0), (torch.float32, torch.bfloat16, 1),
    (torch.bfloat16, torch.bfloat16, 0), (torch.bfloat16, torch.float32, 1)])
def test_merge_kernel_alone(in_dtype, out_dtype, base):
    import context_sharded_mla_gb300 as dcp
    g = torch.Generator().manual_seed(21)
    n, rows = 11, 1000
    o_parts = torch.randn(n, rows, 512, generator=g).to(in_dtype)
    lse_parts = torch.randn(n, rows, generator=g, dtype=torch.float64) * 6
    lse_parts[3, :500] = -math.inf           # empty shards
    lse_parts[:, 7] = -math.inf              # an all-empty row
    o_parts[3, :500] = 0
    dev = "cuda"
    o = torch.empty(rows, 512, dtype=out_dtype, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    dcp.dcp_lse_merge(o_parts.to(dev), lse_parts.to(torch.float32).to(dev), base, o, lse)
    torch.cuda.synchronize()
    ref_o, ref_lse = attention.merge(to_f64(o_parts), to_f64(lse_parts.to(torch.float32)), 2 if base else 0)
    assert_close_o(to_f64(o), ref_o, "merge o")
    assert_close_lse(to_f64(lse), ref_lse, "merge lse")
    assert np.all(to_f64(o)[7] == 0) and math.isinf(float(lse[7]))


def test_single_shard_equals_unsharded():
    """N = 1: the partial is plain attention (checked against the oracle's unsharded form)."""
    cfg = workloads.config("k3", B=2, S=3001, N=1, H=32)
    st = GpuState(cfg)
    o, lse = [to_f64(t) for t in st.decode()]
    for b in range(cfg.B):
        ro, rl = attention.attention(to_f64(st.q[b]), to_f64(st.kv[b]), int(st.S[b]), workloads.SCALE, 2)
        assert_close_o(o[b], ro, "N=1 o")
        assert_close_lse(lse[b], rl, "N=1 lse")


def test_decode_step_with_append():
    """K3-style step: cache holds S-1 tokens, the step appends position S-1 and decodes over S."""
    import context_sharded_mla_gb300 as dcp
    from context_sharded_mla_gb300.step import ShardedMlaDecoder
    cfg = workloads.config("k3", B=3, S=2048 + 5)
    S = workloads.lengths(cfg)
    bt, pool_pages = workloads.block_table(cfg, S)
    dev = "cuda"
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    dec = ShardedMlaDecoder(lay, cfg.B, 1, cfg.H, pool_pages, bt.shape[1], workloads.SCALE, 1)
    kvs = [workloads.gen_kv(cfg, b, int(S[b])) for b in range(cfg.B)]
    btd = bt.to(dev)
    for b in range(cfg.B):
        n = int(S[b]) - 1
        dec.append(kvs[b][:n].to(dev), torch.arange(n, device=dev),
                   torch.full((n,), b, dtype=torch.int32, device=dev), btd)
    q = workloads.gen_q(cfg).to(dev)
    kv_new = torch.stack([kvs[b][-1] for b in range(cfg.B)]).to(dev)
    pos = (S - 1).to(dev)
    req = torch.arange(cfg.B, dtype=torch.int32, device=dev)
    o, lse = dec.step(q, btd, S.to(dev), kv_new, pos, req)
    torch.cuda.synchronize()
    for b in range(cfg.B):
        ro, rl, _, _ = attention.sharded_attention(to_f64(q[b]), to_f64(kvs[b]), int(S[b]), cfg.N, cfg.I,
                                                   workloads.SCALE, 2)
        assert_close_o(to_f64(o[b]), ro, "step o")
        assert_close_lse(to_f64(lse[b]), rl, "step lse")
    assert dec.status_bits() == 0


def test_bad_length_sets_status():
    cfg = workloads.config("tiny", q_len=2, lengths_override=(5,), B=1)
    st = GpuState(cfg)
    st.seq_lens.fill_(1)            # shorter than q_len
    st.decode()
    assert st.dec.status_bits() & 16


def test_extend_more_row_groups_than_clusters():
    """80 causal query tokens x 128 heads = 80 row groups of 128 rows: more groups
    than resident clusters (76 on GB300), run as several waves of stream-K ranges
    with cut units merged by the fixup."""
    cfg = workloads.config("extend", B=2, H=128, q_len=80, S=1500, N=8)
    st = GpuState(cfg)
    _check_state(st, heads=[0, 1, 64, 127])


def test_extend_one_range_per_row_group():
    """76 tokens x 128 heads = 76 row groups: no larger range count gains on 76
    clusters, so each group is one range, no unit is cut and no piece workspace
    is reserved."""
    import context_sharded_mla_gb300 as dcp
    cfg = workloads.config("extend", B=2, H=128, q_len=76, S=1200, N=8)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        ws = dcp.dcp_mla_decode_workspace_size(dcp.Layout(cfg.N, cfg.I, cfg.P), 0, cfg.N, cfg.B, 76, 128)
        assert 0 < ws < 4096            # tile starts only: no piece workspace
        ws80 = dcp.dcp_mla_decode_workspace_size(dcp.Layout(cfg.N, cfg.I, cfg.P), 0, cfg.N, cfg.B, 80, 128)
        assert ws80 > 80 * 128 * 512 * 4  # several ranges per group: pieces reserved
    st = GpuState(cfg)
    _check_state(st, heads=[0, 63, 127])


def test_extend_chunk_across_shard_boundaries():
    """A 200-token chunk with interleave 16 over 4 shards: query rows straddle
    several owner blocks, early rows see fewer shards' tokens."""
    cfg = workloads.config("extend", B=1, H=8, q_len=200, S=1000 + 3, N=4, I=16, P=64)
    st = GpuState(cfg)
    _check_state(st)


def test_extend_at_the_row_limit():
    """q_len * H = 512 x 128 = 65536 query rows, the largest a call takes: 512 row
    groups in waves, causal over a 700-token cache of which 512 are the chunk."""
    cfg = workloads.config("extend", B=1, H=128, q_len=512, S=700, N=4, P=16)
    st = GpuState(cfg)
    _check_state(st, heads=[0, 77, 127])
