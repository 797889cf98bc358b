"""Pins for the oracle's absorption products (no GPU).

The checks come from outside the two einsums: identity 1 (the absorbed score
equals the score against keys up-projected per head, W^UK_h c), identity 2
(full per-head attention with up-projected keys and values equals absorbed
576-d attention followed by the output-side product), permutation weights
(which expose a transposed operand or a mixed-up head), a rank-one closed form,
and a pure-Python triple loop on tiny inputs.
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import absorb, attention

SCALE = 1.0 / math.sqrt(192.0)


def weights(H, seed):
    rng = np.random.default_rng(seed)
    w_kc = rng.standard_normal((H, 128, 512)) / math.sqrt(128)
    w_vc = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    return w_kc, w_vc


@pytest.mark.parametrize("T,H,S", [(1, 1, 5), (3, 4, 17), (2, 7, 64)])
def test_identity1_absorbed_score_equals_unabsorbed(T, H, S):
    rng = np.random.default_rng(T * 100 + H)
    q_nope = rng.standard_normal((T, H, 128))
    q_pe = rng.standard_normal((T, H, 64))
    c = rng.standard_normal((S, 512))
    k_r = rng.standard_normal((S, 64))
    w_kc, _ = weights(H, 5)
    q = absorb.absorbed_query(q_nope, q_pe, w_kc)
    assert q.shape == (T, H, 576)
    latent = np.concatenate([c, k_r], axis=1)
    for h in range(H):
        k_c = c @ w_kc[h].T                          # key of head h: W^UK_h c_t, [S, 128]
        ref = q_nope[:, h] @ k_c.T + q_pe[:, h] @ k_r.T
        assert np.allclose(q[:, h] @ latent.T, ref, rtol=1e-12, atol=1e-11)


@pytest.mark.parametrize("S,H,q_len,base", [(40, 3, 1, 0), (129, 2, 4, 2), (1, 5, 1, 0)])
def test_identity2_full_head_attention(S, H, q_len, base):
    """Per-head attention over up-projected keys and values (the unabsorbed
    form) equals absorbed attention over the shared latent rows, then o @ w_vc."""
    rng = np.random.default_rng(S + H)
    q_nope = rng.standard_normal((q_len, H, 128))
    q_pe = rng.standard_normal((q_len, H, 64))
    c = rng.standard_normal((S + q_len - 1, 512))
    k_r = rng.standard_normal((S + q_len - 1, 64))
    w_kc, w_vc = weights(H, 6)
    total = S + q_len - 1
    q = absorb.absorbed_query(q_nope, q_pe, w_kc)
    o, lse = attention.attention(q, np.concatenate([c, k_r], axis=1), total, SCALE, base)
    got = absorb.absorb_o(o, w_vc)
    assert got.shape == (q_len, H, 128)
    for h in range(H):
        k_c = c @ w_kc[h].T                          # [total, 128]
        v_c = c @ w_vc[h]                            # W^UV_h c_t = (w_vc[h])^T c_t, [total, 128]
        for t in range(q_len):
            vis = S + t                              # causal among the new tokens
            s = SCALE * (k_c[:vis] @ q_nope[t, h] + k_r[:vis] @ q_pe[t, h])
            ref = softmax(s) @ v_c[:vis]
            assert np.allclose(got[t, h], ref, rtol=1e-10, atol=1e-12)
            want_lse = logsumexp(s) / (math.log(2.0) if base == 2 else 1.0)
            assert abs(lse[t, h] - want_lse) < 1e-10


def test_permutation_weights():
    """w_kc[h] scatters q_nope dim k to latent dim pi_h(k); w_vc[h] gathers
    latent dim sigma_h(n) into output dim n.  Different permutations per head."""
    H = 3
    rng = np.random.default_rng(2)
    w_kc = np.zeros((H, 128, 512))
    w_vc = np.zeros((H, 512, 128))
    pis, sigmas = [], []
    for h in range(H):
        pi = rng.permutation(512)[:128]
        sigma = rng.permutation(512)[:128]
        w_kc[h, np.arange(128), pi] = 1.0
        w_vc[h, sigma, np.arange(128)] = 1.0
        pis.append(pi)
        sigmas.append(sigma)
    q_nope = rng.standard_normal((2, H, 128))
    o = rng.standard_normal((2, H, 512))
    q_hat = absorb.absorb_q(q_nope, w_kc)
    v = absorb.absorb_o(o, w_vc)
    for h in range(H):
        want = np.zeros((2, 512))
        want[:, pis[h]] = q_nope[:, h]
        assert np.array_equal(q_hat[:, h], want)
        assert np.array_equal(v[:, h], o[:, h][:, sigmas[h]])


def test_rank_one_closed_form():
    """w_kc[h] = u_h v_h^T gives q_hat = (q . u_h) v_h; w_vc[h] = x_h y_h^T gives (o . x_h) y_h."""
    H = 4
    rng = np.random.default_rng(3)
    u, vv = rng.standard_normal((H, 128)), rng.standard_normal((H, 512))
    x, y = rng.standard_normal((H, 512)), rng.standard_normal((H, 128))
    w_kc = np.einsum("hk,hn->hkn", u, vv)
    w_vc = np.einsum("hk,hn->hkn", x, y)
    q_nope = rng.standard_normal((5, H, 128))
    o = rng.standard_normal((5, H, 512))
    q_hat = absorb.absorb_q(q_nope, w_kc)
    v = absorb.absorb_o(o, w_vc)
    for h in range(H):
        assert np.allclose(q_hat[:, h], np.outer(q_nope[:, h] @ u[h], vv[h]), rtol=1e-12, atol=1e-12)
        assert np.allclose(v[:, h], np.outer(o[:, h] @ x[h], y[h]), rtol=1e-12, atol=1e-12)


def test_bruteforce_tiny():
    """Pure-Python loops over (token, head, out dim, in dim), first 128 dims of 512."""
    T, H = 2, 2
    rng = np.random.default_rng(4)
    q_nope = rng.standard_normal((T, H, 128))
    q_pe = rng.standard_normal((T, H, 64))
    o = rng.standard_normal((T, H, 512))
    w_kc, w_vc = weights(H, 7)
    q = absorb.absorbed_query(q_nope, q_pe, w_kc)
    v = absorb.absorb_o(o, w_vc)
    for t in range(T):
        for h in range(H):
            for n in range(0, 512, 37):
                acc = 0.0
                for k in range(128):
                    acc += float(q_nope[t, h, k]) * float(w_kc[h, k, n])
                assert abs(q[t, h, n] - acc) < 1e-11
            for n in range(128):
                acc = 0.0
                for k in range(512):
                    acc += float(o[t, h, k]) * float(w_vc[h, k, n])
                assert abs(v[t, h, n] - acc) < 1e-11
            assert list(q[t, h, 512:]) == list(q_pe[t, h])


def test_leading_dims_and_empty():
    w_kc, w_vc = weights(3, 8)
    rng = np.random.default_rng(9)
    q_nope = rng.standard_normal((2, 4, 3, 128))       # [B, q_len, H, 128]
    flat = absorb.absorb_q(q_nope.reshape(8, 3, 128), w_kc).reshape(2, 4, 3, 512)
    assert np.array_equal(absorb.absorb_q(q_nope, w_kc), flat)
    assert absorb.absorb_o(np.zeros((0, 3, 512)), w_vc).shape == (0, 3, 128)
