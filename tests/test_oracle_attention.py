"""Pins for the oracle's partial attention and LSE merge (no GPU).

The checks come from outside the oracle: the merge identity (merged shards ==
unsharded attention), closed forms (q = 0, single-token shards, the averaging
counterexample), the monoid laws of the merge operator, the base-e/base-2
identity, a pure-Python triple loop on tiny inputs, and scipy's logsumexp.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention, bruteforce, layout

SCALE = 1.0 / math.sqrt(192.0)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(S, H, q_len, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((q_len, H, 576))
    kv = rng.standard_normal((S, 576))
    return q, kv


@pytest.mark.parametrize("N,I,S,q_len,base", [
    (1, 1, 50, 1, 0), (2, 1, 77, 1, 0), (4, 1, 1024, 1, 0), (8, 1, 333, 1, 2),
    (4, 4, 100, 1, 0), (16, 16, 700, 4, 0), (16, 16, 40, 4, 0), (3, 2, 5, 4, 2), (8, 1, 3, 1, 0)])
def test_merge_equals_unsharded(N, I, S, q_len, base):
    q, kv = rand_case(S, 5, q_len, seed=S + N)
    o, lse, o_p, lse_p = attention.sharded_attention(q, kv, S, N, I, SCALE, base)
    o_ref, lse_ref = attention.attention(q, kv, S, SCALE, base)
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_unsharded_matches_scipy():
    q, kv = rand_case(300, 3, 2, seed=9)
    o, lse = attention.attention(q, kv, 300, SCALE, 0)
    for t in range(2):
        vis = 300 - 2 + t + 1
        s = SCALE * q[t] @ kv[:vis].T
        assert np.allclose(lse[t], logsumexp(s, axis=1), rtol=1e-13)
        assert np.allclose(o[t], softmax(s, axis=1) @ kv[:vis, :512], rtol=1e-11, atol=1e-14)


def test_averaging_counterexample():
    g = json.load(open(os.path.join(GOLDEN, "averaging_counterexample.json")))
    v = g["values"]
    # two shards of one token each: s1 = ln 3, s2 = 0 -> the true output is 3/4
    o_parts = np.array([[[v[0]] * 512], [[v[1]] * 512]])          # [2, 1, 512]
    lse_parts = np.array([[math.log(3.0)], [0.0]])
    o, lse = attention.merge(o_parts, lse_parts, 0)
    assert np.allclose(o, g["case"]["true_output"], rtol=1e-15)
    assert abs(np.mean(o_parts[:, 0, 0]) - g["average_of_local_outputs"]) < 1e-15
    assert abs(lse[0] - math.log(4.0)) < 1e-15
    # the same through the partial: shard 0 holds a token of value 1 scoring ln 3
    q = np.zeros((1, 1, 576))
    q[0, 0, 575] = math.log(3.0) / SCALE
    kv = np.zeros((2, 576))
    kv[0, :512] = 1.0
    kv[0, 575] = 1.0
    o2, lse2, o_p, lse_p = attention.sharded_attention(q, kv, 2, 2, 1, SCALE, 0)
    assert np.allclose(o_p[:, 0, 0, 0], g["local_outputs"])
    assert abs(o2[0, 0, 0] - 0.75) < 1e-12
    # the average of the local outputs differs from the merge for any s1 != s2
    for s1 in (-3.0, -0.5, 0.7, 4.0):
        o3, _ = attention.merge(o_parts, np.array([[s1], [0.0]]), 0)
        assert abs(o3[0, 0] - 1 / (1 + math.exp(-s1))) < 1e-12
        assert abs(o3[0, 0] - 0.5) > 0.1


def test_zero_query_closed_form():
    N, I, S = 4, 2, 203
    rng = np.random.default_rng(4)
    kv = rng.standard_normal((S, 576))
    q = np.zeros((1, 2, 576))
    o, lse, o_p, lse_p = attention.sharded_attention(q, kv, S, N, I, SCALE, 0)
    pos = np.arange(S)
    for r in range(N):
        mine = layout.owner(pos, N, I) == r
        n = mine.sum()
        assert np.allclose(lse_p[r], math.log(n), rtol=1e-14)
        assert np.allclose(o_p[r, 0, 0], kv[mine, :512].mean(axis=0), rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, math.log(S), rtol=1e-14)
    assert np.allclose(o[0, 0], kv[:, :512].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_single_token_shard():
    N, S = 4, 4          # one token per shard
    q, kv = rand_case(S, 3, 1, seed=5)
    _, _, o_p, lse_p = attention.sharded_attention(q, kv, S, N, 1, SCALE, 0)
    for r in range(N):
        s = SCALE * q[0] @ kv[r]
        assert np.allclose(lse_p[r, 0], s, rtol=1e-14)
        assert np.allclose(o_p[r, 0], np.broadcast_to(kv[r, :512], (3, 512)))


def test_empty_shards_identity():
    N, I, S = 8, 1, 3    # shards 3..7 hold nothing
    q, kv = rand_case(S, 2, 1, seed=6)
    o, lse, o_p, lse_p = attention.sharded_attention(q, kv, S, N, I, SCALE, 0)
    for r in range(3, 8):
        assert np.all(np.isneginf(lse_p[r]))
        assert np.all(o_p[r] == 0.0)
    o_ref, lse_ref = attention.attention(q, kv, S, SCALE, 0)
    assert np.allclose(o, o_ref, rtol=1e-13)
    # all-empty rows: o = 0, lse = -inf, no NaN
    o_e, lse_e = attention.merge(np.zeros((3, 2, 512)), np.full((3, 2), -np.inf), 0)
    assert np.all(o_e == 0) and np.all(np.isneginf(lse_e))
    # merging with the unit (0, 0) changes nothing
    o_u, lse_u = attention.merge(np.concatenate([o_p, np.zeros((1,) + o_p.shape[1:])]),
                                 np.concatenate([lse_p, np.full((1,) + lse_p.shape[1:], -np.inf)]), 0)
    assert np.allclose(o_u, o, rtol=1e-15) and np.allclose(lse_u, lse, rtol=1e-15)


def test_merge_monoid_any_tree():
    rng = np.random.default_rng(8)
    n = 7
    o_parts = rng.standard_normal((n, 4, 512))
    lse_parts = rng.normal(0, 5, (n, 4))
    lse_parts[2, 1] = -np.inf
    o_all, lse_all = attention.merge(o_parts, lse_parts, 0)
    for trial in range(20):
        perm = rng.permutation(n)
        items = [(o_parts[i], lse_parts[i]) for i in perm]
        while len(items) > 1:       # random binary tree
            i = int(rng.integers(0, len(items) - 1))
            a, b = items[i], items[i + 1]
            m = attention.merge(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]), 0)
            items[i:i + 2] = [m]
        assert np.allclose(items[0][0], o_all, rtol=1e-12, atol=1e-13)
        assert np.allclose(items[0][1], lse_all, rtol=1e-13)


def test_base2_identity_and_mismatch():
    N, I, S = 4, 1, 257
    q, kv = rand_case(S, 3, 1, seed=10)
    o_e, lse_e, o_pe, lse_pe = attention.sharded_attention(q, kv, S, N, I, SCALE, 0)
    o_2, lse_2, o_p2, lse_p2 = attention.sharded_attention(q, kv, S, N, I, SCALE, 2)
    assert np.allclose(lse_p2, lse_pe * math.log2(math.e), rtol=1e-14)
    assert np.allclose(lse_2, lse_e * math.log2(math.e), rtol=1e-14)
    assert np.allclose(o_2, o_e, rtol=1e-13)
    # base-2 lse merged with base-e weights (a mismatched pair) is wrong
    o_bad, _ = attention.merge(o_p2, lse_p2, 0)
    # make the shard weights unequal first so the mismatch is visible
    lse_skew = lse_pe.copy()
    lse_skew[0] += 3.0
    o_good, _ = attention.merge(o_pe, lse_skew, 0)
    o_mis, _ = attention.merge(o_pe, lse_skew * math.log2(math.e), 0)
    assert np.max(np.abs(o_good - o_mis)) > 1e-3 * np.max(np.abs(o_good))


def test_bruteforce_tiny():
    for (N, I, S, q_len, H) in [(2, 1, 9, 1, 2), (3, 2, 13, 2, 1), (4, 1, 3, 1, 2), (2, 3, 11, 4, 1)]:
        q, kv = rand_case(S, H, q_len, seed=N * 31 + S)
        o_bf, lse_bf, parts_bf = bruteforce.sharded_attention(q.tolist(), kv.tolist(), S, N, I, SCALE)
        o, lse, o_p, lse_p = attention.sharded_attention(q, kv, S, N, I, SCALE, 0)
        assert np.allclose(o, np.array(o_bf), rtol=1e-11, atol=1e-14)
        assert np.allclose(lse, np.array(lse_bf), rtol=1e-12)
        for r in range(N):
            for t in range(q_len):
                for h in range(H):
                    ob, lb = parts_bf[r][t][h]
                    if math.isinf(lb):
                        assert np.isneginf(lse_p[r, t, h]) and np.all(o_p[r, t, h] == 0)
                    else:
                        assert abs(lse_p[r, t, h] - lb) < 1e-11
                        assert np.allclose(o_p[r, t, h], ob, rtol=1e-10, atol=1e-14)


def test_causal_verify_rows():
    """q_len = 4: row t sees exactly positions <= S - 4 + t (checked against a prefix)."""
    S, q_len = 97, 4
    q, kv = rand_case(S, 2, q_len, seed=12)
    o, lse = attention.attention(q, kv, S, SCALE, 0)
    for t in range(q_len):
        o1, lse1 = attention.attention(q[t:t + 1], kv, S - q_len + t + 1, SCALE, 0)
        assert np.allclose(o[t], o1[0], rtol=1e-14) and np.allclose(lse[t], lse1[0], rtol=1e-14)


def test_partial_from_arena_equals_logical():
    N, I, P = 4, 2, 8
    S_list = [61, 5, 0 + 1, 33]
    H, q_len = 3, 2
    B = len(S_list)
    rng = np.random.default_rng(13)
    pages_per = [max(1, -(-s // (N * P))) for s in S_list]
    pool_pages = sum(pages_per) + 2
    perm = rng.permutation(pool_pages)
    bt = np.full((B, max(pages_per)), -1, np.int64)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off:off + n]
        off += n
    arena = np.zeros((N, pool_pages * P, 576), np.uint16)
    kvs = []
    for b, S in enumerate(S_list):
        bits = rng.integers(0, 2**15, size=(S, 576), dtype=np.uint16)  # finite bf16
        bits[:, :] = (bits & 0x3FFF) | 0x3000                           # moderate magnitudes
        kvs.append(bits)
        pos = np.arange(S)
        layout.kv_append(arena, bits, pos, np.full(S, b), bt, N, I, P)
    for b, S in enumerate(S_list):
        q = rng.standard_normal((q_len, H, 576)) if S >= q_len else None
        if q is None:
            continue
        kv = attention.bf16_bits_to_f64(kvs[b])
        for r in range(N):
            oa, la = attention.partial_from_arena(q, arena[r], bt[b], S, r, N, I, P, SCALE, 2)
            ol, ll = attention.partial_logical(q, kv, S, r, N, I, SCALE, 2)
            assert np.array_equal(np.isneginf(la), np.isneginf(ll))
            assert np.allclose(oa, ol, rtol=1e-14, atol=0)
            fin = ~np.isneginf(ll)
            assert np.allclose(la[fin], ll[fin], rtol=1e-14)


def test_bf16_conversion_exact():
    vals = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001], np.uint16)
    f = attention.bf16_bits_to_f64(vals)
    assert f[0] == 1.0 and f[1] == -1.0 and f[3] == 0.0
    assert abs(f[2] - 3.140625) < 1e-15
    assert f[5] == float(np.float32(3.3895314e38))
    assert f[6] == 2.0**-133
