"""A decode step captured in a CUDA graph and replayed.

The pages list CUDA Graph among the things a DCP decode must be validated
under.  The step (slot map, owner-filtered append, partials, merge) is captured
once through the C ABI, then replayed three times with new inputs copied into
the captured buffers (a new query, the next token of every request and the
lengths).  Each replay is checked against the fp64 oracle over the cache as it
stands after that append.

The library's host work per call (argument checks, the stream-K plan, the
tensor maps) depends only on shapes, pointers and the device; every length is
read on the device.  A second test checks a replay bit for bit against the
eager step, then shortens the requests by different amounts and swaps the
query in place: the next replay follows them (checked against the oracle).
"""

import numpy as np

import pytest
import torch

import workloads
from oracle import attention

from harness import GpuState, assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu


def test_decode_step_replays_in_a_cuda_graph():
    import context_sharded_mla_gb300 as dcp
    from context_sharded_mla_gb300.step import ShardedMlaDecoder

    cfg = workloads.config("k3", B=3, H=32, S=3000)
    dev = torch.device("cuda")
    S = workloads.lengths(cfg)
    bt, pool_pages = workloads.block_table(cfg, S)
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    dec = ShardedMlaDecoder(lay, cfg.B, 1, cfg.H, pool_pages, bt.shape[1], workloads.SCALE,
                            dcp.DCP_LSE_BASE_2, torch.float32, device=dev)
    btd = bt.to(dev)
    kv = [workloads.gen_kv(cfg, b, int(S[b])) for b in range(cfg.B)]
    first = int(S[0]) - 3                     # the cache holds S - 3 tokens; three steps append the rest
    for b in range(cfg.B):
        dec.append(kv[b][:first].to(dev), torch.arange(first, device=dev),
                   torch.full((first,), b, dtype=torch.int32, device=dev), btd)
    q_s = torch.empty(cfg.B, 1, cfg.H, 576, dtype=torch.bfloat16, device=dev)
    kv_s = torch.empty(cfg.B, 576, dtype=torch.bfloat16, device=dev)
    pos_s = torch.empty(cfg.B, dtype=torch.int64, device=dev)
    req_s = torch.arange(cfg.B, dtype=torch.int32, device=dev)
    len_s = torch.empty(cfg.B, dtype=torch.int64, device=dev)
    qs = []

    def load_step(k):
        g = torch.Generator().manual_seed(100 + k)
        q = torch.randn(cfg.B, 1, cfg.H, 576, generator=g).to(torch.bfloat16)
        qs.append(q)
        q_s.copy_(q.to(dev))
        kv_s.copy_(torch.stack([kv[b][first + k] for b in range(cfg.B)]).to(dev))
        pos_s.fill_(first + k)
        len_s.fill_(first + k + 1)

    def check(k):
        torch.cuda.synchronize()
        n = first + k + 1
        o = to_f64(dec.o)
        lse = to_f64(dec.lse)
        for b in range(cfg.B):
            ref_o, ref_lse, _, _ = attention.sharded_attention(to_f64(qs[k][b]), to_f64(kv[b][:n]), n, cfg.N, cfg.I,
                                                               workloads.SCALE, cfg.base)
            assert_close_o(o[b], ref_o, f"graph step {k} b={b}")
            assert_close_lse(lse[b], ref_lse, f"graph step {k} b={b}")
        assert dec.status_bits() == 0

    # step 0 runs eagerly on a side stream (warm-up before capture), then is captured
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    load_step(0)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        dec.step(q_s, btd, len_s, kv_s, pos_s, req_s)
    torch.cuda.current_stream().wait_stream(side)
    check(0)
    graph = torch.cuda.CUDAGraph()
    launches0 = dcp.dcp_launch_count()
    with torch.cuda.graph(graph):
        dec.step(q_s, btd, len_s, kv_s, pos_s, req_s)
    captured = dcp.dcp_launch_count() - launches0
    assert captured >= 4                      # append, plan, partial, (fixup,) merge
    for k in (1, 2):
        load_step(k)
        graph.replay()
        check(k)
    # the captured launches ran on replay, not at capture time: replaying step 2
    # again (same slot, same row) gives the same result
    graph.replay()
    check(2)


def test_replay_is_bit_exact_and_follows_shorter_lengths():
    cfg = workloads.config("k3", B=3, S=3000 + 11, seed=31)
    st = GpuState(cfg)
    dec = st.dec
    dev = st.q.device
    q = st.q.clone()
    seq = st.seq_lens.clone()
    # each replay re-appends every request's last token (the same bytes to the same slot)
    last = (st.S - 1).to(dev)
    kv_last = torch.stack([st.kv[b][int(st.S[b]) - 1] for b in range(cfg.B)]).to(dev)
    req = torch.arange(cfg.B, dtype=torch.int32, device=dev)

    o_e, lse_e = dec.step(q, st.bt, seq, kv_last, last, req)
    torch.cuda.synchronize()
    o_e, lse_e = o_e.clone(), lse_e.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                   # warm-up on a side stream, as capture wants
        for _ in range(2):
            dec.step(q, st.bt, seq, kv_last, last, req)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        o_g, lse_g = dec.step(q, st.bt, seq, kv_last, last, req)
    graph.replay()
    torch.cuda.synchronize()
    assert dec.status_bits() == 0
    assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e), "replay differs from the eager step"

    # new lengths and a new query, written in place; the replay follows them
    S_new = st.S - torch.tensor([1, 777, 2048], dtype=st.S.dtype)
    g = torch.Generator().manual_seed(77)
    q_new = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    seq.copy_(S_new.to(dev))
    q.copy_(q_new.to(dev))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert dec.status_bits() == 0
    for b in range(cfg.B):
        o_ref, l_ref, _op, _lp = attention.sharded_attention(to_f64(q_new[b]), to_f64(st.kv[b]), int(S_new[b]),
                                                             cfg.N, cfg.I, workloads.SCALE, cfg.base)
        assert_close_o(to_f64(o_g[b]), o_ref, f"replay with new lengths b={b}")
        assert_close_lse(to_f64(lse_g[b]), l_ref, f"replay with new lengths b={b}")
    assert not np.array_equal(to_f64(o_g), to_f64(o_e))
