"""Oracle: the cross-rank exchange of the partials and the two merge strategies.

TEST INFRASTRUCTURE ONLY (see the package docstring).  fp64 arithmetic.

With W ranks (one GPU each), rank w holds the context shards
[w*N/W, (w+1)*N/W) and is the "head owner" of heads [d*H/W, (d+1)*H/W) for
d = w.  Every rank attends all H heads against its own shards (the query is
replicated or all-gathered), so after the partial step rank w holds
(o_r, lse_r) for its shards and ALL heads; the exchange hands each head owner
the partials of its heads from every shard, and it merges them.

Sources
-------
* "Decode Context Parallelism" (zdszero), section "通信策略":
  - "合并：All-to-All": each rank cuts O_r by head into N pieces and sends each
    piece, together with the matching LSE in the same buffer, in one
    all-to-all to the rank that finally owns those heads; the receiver then
    holds, for its own heads, the partials of every shard and merges them
    locally with the LSE rule.
  - "合并：AllGather + ReduceScatter": all-gather the LSE of every rank; each
    rank computes the global L and corrects its own partial to
    exp(L_r - L) * O_r; a reduce-scatter then sums those corrected partials and
    scatters the result by head.
  - Same page, "Core abstraction" / "Theory": the merge identity used here.
* "MLA 的 Decode Context Parallelism", section 4, stages 6-7 (all-to-all of
  (o^(r), lse_r) to the head owner; two-pass LSE merge there) and section 5
  (the all-to-all carries B*H*(512 + 4)*2 bytes per rank and step: bf16 o and
  an fp32 lse, about 6.3 MB at B=64, H=96, of which 7/8 leaves the rank).

Readings (the pages assume one shard per rank and H divisible by the group):
* With N > W, rank w holds N/W consecutive shards and sends all of them; parts
  reach the receiver in shard order.  N % W == 0 and H % W == 0 are required.
* Wire format of one rank's all-to-all send buffer (the library's format, so the
  byte layout has a definition to compare with): for each destination d in
  order, an o block [n_held, T, H/W, 512] in the wire dtype (bf16 rounded to
  nearest even, or f32) followed by an lse block [n_held, T, H/W] f32, the two
  padded with zero bytes to a multiple of 256 bytes (so that every chunk starts
  aligned), where T is the number of query tokens (B * q_len) and n_held = N / W.
"""

from __future__ import annotations

import numpy as np

from .attention import merge


def shard_range(w: int, N: int, W: int):
    """Shards [begin, end) held by rank w of W (N % W == 0)."""
    if W < 1 or N % W:
        raise ValueError(f"{N} shards do not split evenly over {W} ranks")
    n = N // W
    return w * n, (w + 1) * n


def head_range(d: int, H: int, W: int):
    """Heads [begin, end) owned by rank d of W after the exchange (H % W == 0)."""
    if W < 1 or H % W:
        raise ValueError(f"{H} heads do not split evenly over {W} ranks")
    n = H // W
    return d * n, (d + 1) * n


def a2a_received(o_parts, lse_parts, W: int):
    """What each head owner holds after the all-to-all.

    o_parts [N, T, H, 512], lse_parts [N, T, H]: every shard's partials (all
    heads).  Returns a list over d of (o [N, T, H/W, 512], lse [N, T, H/W]):
    head slice d of every shard, shards in order (rank w's shards come from
    rank w).
    """
    o_parts = np.asarray(o_parts)
    lse_parts = np.asarray(lse_parts)
    N, _T, H = lse_parts.shape
    out = []
    for d in range(W):
        h0, h1 = head_range(d, H, W)
        o_d = np.concatenate([o_parts[slice(*shard_range(w, N, W)), :, h0:h1] for w in range(W)])
        l_d = np.concatenate([lse_parts[slice(*shard_range(w, N, W)), :, h0:h1] for w in range(W)])
        out.append((o_d, l_d))
    return out


def a2a_merge(o_parts, lse_parts, W: int, base=0):
    """The all-to-all strategy end to end: per head owner d, the LSE merge of
    the N partials it received.  Returns a list over d of (o [T, H/W, 512], lse [T, H/W])."""
    return [merge(o_d, l_d, base) for o_d, l_d in a2a_received(o_parts, lse_parts, W)]


def global_lse(lse_all, base=0):
    """Step 1 of AllGather + ReduceScatter: from the gathered lse of all N shards
    [N, ...], L = m + log sum_r exp(lse_r - m) (log2 / exp2 in base 2); rows
    whose shards are all empty get -inf."""
    base = 2 if base in (1, 2) else 0
    lse_all = np.asarray(lse_all, dtype=np.float64)
    m = lse_all.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    pw = np.exp2 if base == 2 else np.exp
    Z = np.where(empty, 1.0, pw(lse_all - m_safe).sum(axis=0))
    return np.where(empty, -np.inf, m_safe + (np.log2(Z) if base == 2 else np.log(Z)))


def rescale_local(lse_all, o_held, shard_begin: int, W: int, base=0):
    """Step 2 on one rank: sum over its held shards s of exp(lse_s - L) * O_s
    (2 ** (lse_s - L) in base 2; an empty shard contributes 0), with L from
    global_lse.  lse_all [N, T, H] (every shard), o_held [n_held, T, H, 512].
    Returned head-sliced for the reduce-scatter: (o_sum [W, T, H/W, 512],
    L [W, T, H/W]); block d holds heads [d*H/W, (d+1)*H/W)."""
    base = 2 if base in (1, 2) else 0
    lse_all = np.asarray(lse_all, dtype=np.float64)
    o_held = np.asarray(o_held, dtype=np.float64)
    n_held = o_held.shape[0]
    L = global_lse(lse_all, base)
    L_safe = np.where(np.isneginf(L), 0.0, L)
    pw = np.exp2 if base == 2 else np.exp
    wgt = pw(lse_all[shard_begin:shard_begin + n_held] - L_safe)   # exp(-inf) = 0 for an empty shard
    total = (wgt[..., None] * o_held).sum(axis=0)
    total = np.where(np.isneginf(L)[..., None], 0.0, total)
    H = lse_all.shape[2]
    blocks = [head_range(d, H, W) for d in range(W)]
    return (np.stack([total[:, h0:h1] for h0, h1 in blocks]), np.stack([L[:, h0:h1] for h0, h1 in blocks]))


def ag_rs_merge(o_parts, lse_parts, W: int, base=0):
    """The AllGather + ReduceScatter strategy end to end.

    1. all-gather: every rank sees lse_r of all N shards and forms the global L
       (global_lse);
    2. each rank w corrects its own shards (rescale_local);
    3. reduce-scatter: the ranks' corrected sums are added and rank d keeps heads
       [d*H/W, (d+1)*H/W).
    Returns a list over d of (o [T, H/W, 512], lse [T, H/W]).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    N = lse_parts.shape[0]
    sums, L = None, None
    for w in range(W):
        s0, s1 = shard_range(w, N, W)
        o_sum, L = rescale_local(lse_parts, o_parts[s0:s1], s0, W, base)
        sums = o_sum if sums is None else sums + o_sum
    return [(sums[d], L[d]) for d in range(W)]


def to_bf16_bits(x):
    """Round to the nearest bf16 (ties to even) via fp32; returns uint16 bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), r)


def pack(o_held, lse_held, W: int, wire_bf16: bool):
    """One rank's all-to-all send buffer in the wire format (module docstring).

    o_held [n_held, T, H, 512], lse_held [n_held, T, H] (this rank's shards, all
    heads).  Returns uint8 [W, chunk_bytes]: row d goes to rank d.
    """
    o_held = np.asarray(o_held)
    lse_held = np.asarray(lse_held)
    _n, _T, H = lse_held.shape
    chunks = []
    for d in range(W):
        h0, h1 = head_range(d, H, W)
        o = o_held[:, :, h0:h1]
        ob = to_bf16_bits(o).tobytes() if wire_bf16 else np.asarray(o, np.float32).tobytes()
        lb = np.ascontiguousarray(lse_held[:, :, h0:h1], dtype=np.float32).tobytes()
        pad = bytes(-(len(ob) + len(lb)) % 256)
        chunks.append(np.frombuffer(ob + lb + pad, dtype=np.uint8))
    return np.stack(chunks)


def chunk_bytes(n_held: int, T: int, H: int, W: int, wire_bf16: bool) -> int:
    """Bytes one rank sends to each rank: n_held * T * (H/W) * (512 * e + 4),
    rounded up to a multiple of 256."""
    hd = head_range(0, H, W)[1]
    n = n_held * T * hd * (512 * (2 if wire_bf16 else 4) + 4)
    return n + (-n % 256)


def unpack(recv, n_held: int, T: int, H: int, W: int, wire_bf16: bool):
    """Inverse of the wire format for one receiver: recv uint8 [W, chunk_bytes]
    (row w came from rank w) -> (o [W * n_held, T, H/W, 512] fp64, lse [W * n_held, T, H/W])."""
    hd = H // W
    recv = np.asarray(recv, dtype=np.uint8).reshape(W, -1)
    n_o = n_held * T * hd * 512
    ob = n_o * (2 if wire_bf16 else 4)
    os_, ls_ = [], []
    for w in range(W):
        raw = recv[w].tobytes()
        if wire_bf16:
            bits = np.frombuffer(raw[:ob], dtype=np.uint16)
            o = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        else:
            o = np.frombuffer(raw[:ob], dtype=np.float32)
        os_.append(o.astype(np.float64).reshape(n_held, T, hd, 512))
        ls_.append(np.frombuffer(raw[ob:ob + 4 * n_held * T * hd], dtype=np.float32).astype(np.float64)
                   .reshape(n_held, T, hd))
    return np.concatenate(os_), np.concatenate(ls_)


def merge_received(recv, n_held: int, T: int, H: int, W: int, wire_bf16: bool, base=0):
    """The receiver's local LSE merge of an all-to-all receive buffer."""
    o, lse = unpack(recv, n_held, T, H, W, wire_bf16)
    return merge(o, lse, base)
