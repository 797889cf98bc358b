"""Oracle pins: pure-Python loop versions for tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

These are written a second way on purpose, so that a mistake in ``layout`` or
``attention`` shows up as a disagreement:

* ownership is found by dealing blocks of I consecutive positions to shards
  0, 1, ..., N-1 in turn and appending each dealt position to its shard's list
  ("PCP / DCP：计算、KV 布局与块轮转", sections 5 and 6: token RR and block RR
  keep each rank's tokens compact in arrival order); the local row is the index
  in that list, and count is the length of the list after x positions;
* attention is a triple loop with math.exp, one score at a time, and the merge
  is the un-shifted ratio sum_r Z_r O_r / sum_r Z_r of the derivation in
  "Decode Context Parallelism" (zdszero), "Theory".
"""

from __future__ import annotations

import math


def deal(S, N, I):
    """Lists of positions held by each shard after dealing S positions."""
    lists = [[] for _ in range(N)]
    shard = 0
    p = 0
    while p < S:
        for _ in range(I):
            if p >= S:
                break
            lists[shard].append(p)
            p += 1
        shard = (shard + 1) % N
    return lists


def owner_row_table(S, N, I):
    """{p: (owner, local row)} for p < S, from the dealt lists."""
    table = {}
    for r, lst in enumerate(deal(S, N, I)):
        for row, p in enumerate(lst):
            table[p] = (r, row)
    return table


def count(r, x, N, I):
    return len(deal(x, N, I)[r])


def attend(q_row, keys, scale):
    """Z = sum exp(s), N = sum exp(s) v over `keys` (lists of 576 floats)."""
    Z = 0.0
    acc = [0.0] * 512
    for k in keys:
        s = scale * sum(a * b for a, b in zip(q_row, k))
        e = math.exp(s)
        Z += e
        for d in range(512):
            acc[d] += e * k[d]
    return Z, acc


def sharded_attention(q, kv, S, N, I, scale):
    """Merged output of one request by loops: q [q_len][H][576], kv [S][576].

    Returns (o [q_len][H][512], lse [q_len][H], per-shard (o_r, lse_r)), lse base e.
    """
    q_len = len(q)
    H = len(q[0])
    lists = deal(S, N, I)
    o = [[None] * H for _ in range(q_len)]
    lse = [[None] * H for _ in range(q_len)]
    shard_parts = [[[None] * H for _ in range(q_len)] for _ in range(N)]
    for t in range(q_len):
        pos_t = S - q_len + t
        for h in range(H):
            Ztot = 0.0
            Ntot = [0.0] * 512
            for r in range(N):
                keys = [kv[p] for p in lists[r] if p <= pos_t]
                Z, acc = attend(q[t][h], keys, scale)
                if Z > 0:
                    shard_parts[r][t][h] = ([a / Z for a in acc], math.log(Z))
                else:
                    shard_parts[r][t][h] = ([0.0] * 512, -math.inf)
                Ztot += Z
                Ntot = [a + b for a, b in zip(Ntot, acc)]
            if Ztot > 0:
                o[t][h] = [a / Ztot for a in Ntot]
                lse[t][h] = math.log(Ztot)
            else:
                o[t][h] = [0.0] * 512
                lse[t][h] = -math.inf
    return o, lse, shard_parts
