"""Pins for the oracle's cross-rank exchange (no GPU).

The checks come from outside the exchange code: the merge identity (what every
head owner ends with equals unsharded attention of its heads), the two
strategies of the "通信策略" section agreeing with each other, a labelled
brute-force bijection of (shard, head) pairs, the page's byte accounting of
the all-to-all, the averaging counterexample pushed through both strategies,
torch's bf16 rounding for the wire dtype, and rows whose shards are all empty.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention, exchange

SCALE = 1.0 / math.sqrt(192.0)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(S, H, q_len, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((q_len, H, 576)), rng.standard_normal((S, 576))


@pytest.mark.parametrize("N,W,I,S,q_len,H,base", [
    (8, 8, 1, 333, 1, 8, 2), (8, 2, 1, 500, 1, 6, 0), (8, 4, 1, 41, 2, 4, 0), (4, 1, 1, 64, 1, 3, 0),
    (16, 4, 16, 700, 4, 8, 0), (16, 8, 16, 40, 4, 8, 2), (2, 2, 1, 1, 1, 2, 0)])
def test_both_strategies_equal_unsharded_attention(N, W, I, S, q_len, H, base):
    q, kv = rand_case(S, H, q_len, seed=S * 7 + N + W)
    _o, _l, o_p, l_p = attention.sharded_attention(q, kv, S, N, I, SCALE, base)
    o_ref, l_ref = attention.attention(q, kv, S, SCALE, base)
    a2a = exchange.a2a_merge(o_p, l_p, W, base)
    agrs = exchange.ag_rs_merge(o_p, l_p, W, base)
    for d in range(W):
        h0, h1 = exchange.head_range(d, H, W)
        assert np.allclose(a2a[d][0], o_ref[:, h0:h1], rtol=1e-12, atol=1e-14)
        assert np.allclose(a2a[d][1], l_ref[:, h0:h1], rtol=1e-12, atol=1e-12)
        assert np.allclose(agrs[d][0], o_ref[:, h0:h1], rtol=1e-12, atol=1e-14)
        assert np.allclose(agrs[d][1], l_ref[:, h0:h1], rtol=1e-12, atol=1e-12)


def test_received_parts_are_a_bijection_of_shard_head_pairs():
    N, W, T, H = 8, 4, 3, 8
    # label every partial row with (shard, token, head) and check where it lands
    o_p = np.zeros((N, T, H, 512))
    l_p = np.zeros((N, T, H))
    for r in range(N):
        for t in range(T):
            for h in range(H):
                o_p[r, t, h, :] = 1e6 * r + 1e3 * t + h
                l_p[r, t, h] = 1e6 * r + 1e3 * t + h
    seen = set()
    for d, (o_d, l_d) in enumerate(exchange.a2a_received(o_p, l_p, W)):
        assert o_d.shape == (N, T, H // W, 512) and l_d.shape == (N, T, H // W)
        for k in range(N):
            for t in range(T):
                for hh in range(H // W):
                    code = l_d[k, t, hh]
                    r, rest = divmod(int(code), 10**6)
                    tt, h = divmod(rest, 10**3)
                    assert (r, tt, h) == (k, t, d * (H // W) + hh)   # shard order, own heads
                    assert np.all(o_d[k, t, hh] == code)             # o travels with its lse
                    seen.add((r, tt, h))
    assert len(seen) == N * T * H


def test_wire_bytes_match_the_page_accounting():
    g = json.load(open(os.path.join(GOLDEN, "mla_accounting.json")))
    # K3 step: B=64, H=96, one shard per rank on 8 ranks, bf16 o + fp32 lse
    # The page's formula gives the lse four 2-byte slots, (512 + 4) x 2 B per row;
    # this wire format carries one fp32 lse, 512 x 2 + 4 B.  Both round to the
    # page's printed figures.
    per_dest = exchange.chunk_bytes(1, 64, 96, 8, True)
    total = per_dest * 8
    assert total == 64 * 96 * (512 * 2 + 4)
    assert total <= 64 * 96 * (512 + 4) * 2
    assert abs(total / 1e6 - g["a2a_partials"]["approx_MB"]) < 0.05
    assert abs(total * 7 / 8 / 1e6 - g["a2a_partials"]["sent_per_rank_MB"]) < 0.06
    rng = np.random.default_rng(3)
    buf = exchange.pack(rng.standard_normal((1, 64, 96, 512)), rng.standard_normal((1, 64, 96)), 8, True)
    assert buf.shape == (8, per_dest)
    # a chunk that is not a multiple of 256 bytes is padded with zeros
    assert exchange.chunk_bytes(2, 5, 8, 4, True) == 20736 > 2 * 5 * 2 * (1024 + 4)
    buf = exchange.pack(rng.standard_normal((2, 5, 8, 512)), rng.standard_normal((2, 5, 8)), 4, True)
    assert buf.shape == (4, 20736) and not buf[:, 2 * 5 * 2 * 1028:].any()


@pytest.mark.parametrize("wire_bf16", [False, True])
def test_pack_then_unpack_per_receiver(wire_bf16):
    N, W, T, H = 8, 4, 5, 8
    n = N // W
    rng = np.random.default_rng(5)
    o_p = rng.standard_normal((N, T, H, 512))
    l_p = rng.standard_normal((N, T, H))
    l_p[3, 1, :] = -np.inf                                   # an empty shard travels as -inf
    sends = [exchange.pack(o_p[w * n:(w + 1) * n], l_p[w * n:(w + 1) * n], W, wire_bf16) for w in range(W)]
    for d in range(W):
        recv = np.stack([sends[w][d] for w in range(W)])     # the all-to-all: row w came from rank w
        o_d, l_d = exchange.unpack(recv, n, T, H, W, wire_bf16)
        h0, h1 = exchange.head_range(d, H, W)
        want_o = o_p[:, :, h0:h1]
        if wire_bf16:
            want_o = torch.from_numpy(want_o).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
        else:
            want_o = want_o.astype(np.float32).astype(np.float64)
        assert np.array_equal(o_d, want_o)
        assert np.array_equal(l_d, l_p[:, :, h0:h1].astype(np.float32).astype(np.float64))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(100000) * 10 ** rng.uniform(-30, 30, 100000),
                        [0.0, -0.0, np.inf, -np.inf, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895e38]]).astype(np.float32)
    got = exchange.to_bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert exchange.to_bf16_bits(np.array([np.nan], np.float32))[0] & 0x7FFF > 0x7F80


def test_averaging_counterexample_through_both_strategies():
    g = json.load(open(os.path.join(GOLDEN, "averaging_counterexample.json")))
    # two shards of one token each on two ranks, two heads (identical), s1 = ln 3, s2 = 0
    v = g["values"]
    o_p = np.array([[[[v[0]] * 512] * 2], [[[v[1]] * 512] * 2]], dtype=np.float64)   # [2, 1, 2, 512]
    l_p = np.array([[[math.log(3.0)] * 2], [[0.0] * 2]])
    for res in (exchange.a2a_merge(o_p, l_p, 2, 0), exchange.ag_rs_merge(o_p, l_p, 2, 0)):
        for d in range(2):
            assert np.allclose(res[d][0], g["case"]["true_output"], rtol=1e-15)
            assert abs(res[d][0][0, 0, 0] - g["average_of_local_outputs"]) > 0.2


@pytest.mark.parametrize("base", [0, 2])
def test_all_empty_rows(base):
    N, W, T, H = 4, 2, 2, 4
    rng = np.random.default_rng(1)
    o_p = rng.standard_normal((N, T, H, 512))
    l_p = rng.standard_normal((N, T, H))
    o_p[:, 1] = 0.0
    l_p[:, 1] = -np.inf                                      # token 1 sees no shard at all
    l_p[2, 0] = -np.inf
    o_p[2, 0] = 0.0                                          # shard 2 empty for token 0
    ref_o, ref_l = attention.merge(o_p, l_p, base)
    for res in (exchange.a2a_merge(o_p, l_p, W, base), exchange.ag_rs_merge(o_p, l_p, W, base)):
        for d in range(W):
            h0, h1 = exchange.head_range(d, H, W)
            assert np.all(res[d][0][1] == 0.0) and np.all(np.isneginf(res[d][1][1]))
            assert np.allclose(res[d][0], ref_o[:, h0:h1], rtol=1e-12, atol=1e-14)
            assert np.array_equal(np.isneginf(res[d][1]), np.isneginf(ref_l[:, h0:h1]))


def test_uneven_splits_are_rejected():
    with pytest.raises(ValueError):
        exchange.shard_range(0, 6, 4)
    with pytest.raises(ValueError):
        exchange.head_range(0, 10, 4)
