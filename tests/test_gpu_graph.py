"""A decode step captured as a CUDA graph and replayed, against eager calls and the oracle.

The library's host work for a call (argument checks, the stream-K plan, the
tensor maps) depends only on shapes, pointers and the device; every sequence
length is read on the device, where the plan kernel turns the lengths into the
ranges' tile counts.  So a captured step (append + partials + merge) replays
correctly after the lengths, the queries or the cache change in place, with no
host work per step.  The test captures a step, checks a replay bit for bit
against the eager call, then shortens the requests and swaps the query in place
and checks the next replay against the oracle.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention

from harness import GpuState, assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu


def test_step_graph_replay_matches_eager_and_oracle():
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
