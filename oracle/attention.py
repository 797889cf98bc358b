"""Oracle: per-shard partial attention, the exact LSE merge, unsharded attention.

TEST INFRASTRUCTURE ONLY (see the package docstring).  All arithmetic in fp64.

Shapes: one request at a time.
  q      [q_len, H, 576]  absorbed query rows [q_hat_C (512) || q_R (64)]
  kv     [S, 576]         latent rows [c_K (512) || k_R (64)] in position order
  o      [q_len, H, 512]  values live in the first 512 dims of a latent row
  lse    [q_len, H]

Sources
-------
* "MLA 的 Decode Context Parallelism", section 2 (absorbed form): decode is a
  576-d single-KV-head MQA; the query of each head is [q_hat_C || q_R]; the
  cache row is [c_K || k_R]; the value is c_K (512 dims), so the scores use all
  576 dims and the output uses dims 0..511 of the same row.
* "Decode Context Parallelism" (zdszero), "Core abstraction" idea 2 and
  "Theory / derivation": O_r = softmax_local(q k^T / sqrt(D)) V_r and
  L_r = log sum_{p in P_r} exp(s_p); merged O = sum_r exp(L_r) O_r / sum_r exp(L_r);
  stable form with m = max_r L_r; L = m + log sum_r exp(L_r - m); the exp/log
  pair must match the base the kernel reports (e or 2).
* "PCP / DCP：计算、KV 布局与块轮转", section 4.1: an empty shard contributes a
  zero-weight state (the unit (Z, N) = (0, 0) of the merge operator):
  lse = -inf and o = 0.
* SGLang "Decode context parallelism", "DCP x speculative decoding": the verify
  path passes global KV lengths so causality sees the whole sequence.  Reading:
  with S_b tokens cached (the q_len new ones included), query row t sits at
  position S_b - q_len + t and sees positions p <= S_b - q_len + t.
"""

from __future__ import annotations

import math

import numpy as np

from . import layout

LN2 = math.log(2.0)


def bf16_bits_to_f64(bits):
    """Exact bf16 -> fp64: a bf16 bit pattern is the top half of an fp32."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _softmax_attend(q_rows, K, scale, base):
    """Two-pass softmax attention of q_rows [R, 576] over K [n, 576].

    Returns (o [R, 512], lse [R]) with lse in the requested base; an empty K
    gives o = 0, lse = -inf.
    """
    R = q_rows.shape[0]
    if K.shape[0] == 0:
        return np.zeros((R, 512)), np.full(R, -np.inf)
    s = scale * (q_rows @ K.T)                 # scores over all 576 dims
    m = s.max(axis=1, keepdims=True)           # pass 1: row maximum
    e = np.exp(s - m)                          # pass 2: shifted exponentials
    Z = e.sum(axis=1)
    o = (e @ K[:, :512]) / Z[:, None]          # values = first 512 dims
    lse = m[:, 0] + np.log(Z)                  # natural-log LSE
    if base == 2:
        lse = lse / LN2                        # log2 Z = ln Z / ln 2
    return o, lse


def query_positions(S, q_len):
    """Positions of the q_len new query tokens of a request holding S tokens."""
    return np.arange(S - q_len, S, dtype=np.int64)


def partial_logical(q, kv, S, r, N, I, scale, base=0):
    """(o_r, lse_r) of shard r, from the request's KV in position order.

    The visible set of query row t is {p < S : owner(p) = r, p <= pos_t}.
    base: 0 -> natural log, 2 (or 1) -> log2 of the same sum.
    """
    base = 2 if base in (1, 2) else 0
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    q_len, H, _ = q.shape
    pos = np.arange(S, dtype=np.int64)
    mine = layout.owner(pos, N, I) == r
    o = np.zeros((q_len, H, 512))
    lse = np.full((q_len, H), -np.inf)
    for t, pos_t in enumerate(query_positions(S, q_len)):
        vis = mine & (pos <= pos_t)
        o[t], lse[t] = _softmax_attend(q[t], kv[:S][vis], scale, base)
    return o, lse


def partial_from_arena(q, arena_r_bits, bt_row, S, r, N, I, P, scale, base=0):
    """(o_r, lse_r) of shard r, reading shard r's own pool through the block table.

    Local rows 0 .. count_r(S)-1 hold shard r's tokens in position order; local
    row rho is at slot bt_row[rho // P] * P + rho % P of the pool and holds the
    global position global_pos(r, rho).
    """
    base = 2 if base in (1, 2) else 0
    q = np.asarray(q, dtype=np.float64)
    q_len, H, _ = q.shape
    n = int(layout.count(r, S, N, I))
    rows = np.arange(n, dtype=np.int64)
    p = layout.global_pos(r, rows, N, I)
    slots = layout.physical_slot(bt_row, rows, P) if n else np.zeros(0, np.int64)
    K = bf16_bits_to_f64(np.asarray(arena_r_bits)[slots]) if n else np.zeros((0, 576))
    o = np.zeros((q_len, H, 512))
    lse = np.full((q_len, H), -np.inf)
    for t, pos_t in enumerate(query_positions(S, q_len)):
        vis = p <= pos_t
        o[t], lse[t] = _softmax_attend(q[t], K[vis], scale, base)
    return o, lse


def merge(o_parts, lse_parts, base=0):
    """Exact LSE merge of n partials.

    o_parts [n, ..., 512], lse_parts [n, ...] (all in the same base).
    m = max_r lse_r; w_r = exp(lse_r - m) (2**(lse_r - m) in base 2);
    lse = m + log(sum w) (log2 in base 2); o = sum_r w_r o_r / sum_r w_r.
    Rows whose partials are all empty give o = 0, lse = -inf.
    """
    base = 2 if base in (1, 2) else 0
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    d = lse_parts - m_safe
    w = np.exp2(d) if base == 2 else np.exp(d)        # exp(-inf) = 0 for empty shards
    Zs = w.sum(axis=0)
    Zs_safe = np.where(empty, 1.0, Zs)
    lse = m_safe + (np.log2(Zs_safe) if base == 2 else np.log(Zs_safe))
    lse = np.where(empty, -np.inf, lse)
    o = (w[..., None] * o_parts).sum(axis=0) / Zs_safe[..., None]
    o = np.where(empty[..., None], 0.0, o)
    return o, lse


def attention(q, kv, S, scale, base=0):
    """Unsharded attention of the q_len query rows over all visible positions."""
    base = 2 if base in (1, 2) else 0
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    q_len, H, _ = q.shape
    o = np.zeros((q_len, H, 512))
    lse = np.full((q_len, H), -np.inf)
    for t, pos_t in enumerate(query_positions(S, q_len)):
        o[t], lse[t] = _softmax_attend(q[t], kv[: pos_t + 1], scale, base)
    return o, lse


def sharded_attention(q, kv, S, N, I, scale, base=0):
    """All N partials of one request and their merge: (o, lse, o_parts, lse_parts)."""
    parts = [partial_logical(q, kv, S, r, N, I, scale, base) for r in range(N)]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    o, lse = merge(o_parts, lse_parts, base)
    return o, lse, o_parts, lse_parts
