"""Oracle: slot mapping, chunk share and owner-filtered append (fp64/int64, CPU).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Notation: N shards, I interleave (block) size, P physical page size, positions
are request-global token positions p >= 0.

Sources
-------
* "Decode Context Parallelism" (zdszero), "Core abstraction", idea 1:
  owner(p) = p mod N, row(p) = floor(p / N); a chunk [a, a+L) gives shard r the
  share count(a+L) - count(a), count(x) = #{p < x : p owned by r}.
* "PCP / DCP：计算、KV 布局与块轮转", section 6 "Block RR":
  owner(t) = (t // B) % P_dcp, local_index(t) = (t // (B * P_dcp)) * B + t % B,
  local_len(N, r) = (N // (P_dcp * B)) * B + clamp(N % (P_dcp * B) - r * B, 0, B).
  (That page writes the DCP size as P and the block size as B; here the DCP
  size is N and the block size is the interleave I.)  B = 1 is token RR.
* Same page, section "KV cache 管理": slot = page_id * page_size + offset_in_page.
* vLLM-Ascend "上下文并行（CP）", section "块表": virtual_block_size =
  block_size * cp_size; block index x // vbs; offset x % vbs; local block index
  offset // interleave; rank = local block index % cp_size; offset in the local
  block = (local block index // cp_size) * interleave + offset % interleave;
  requires block_size % interleave == 0.
* SGLang "Decode context parallelism", "Virtual KV layout": every rank sees the
  same request-to-token map and one widened virtual page maps to one physical
  page on each rank.  Reading used here: one block table per request, shared by
  all shards; shard r keeps its local row rho at bt[b][rho // P] * P + rho % P
  of its own pool.
* "PCP / DCP：计算、KV 布局与块轮转", section "PD + DCP：从完整源页抽取本
  rank 的 token": a request prefilled without DCP (full pages) is moved to a
  DCP decode instance; rank r keeps the tokens whose request position it owns
  (selected by request position, never by physical slot), reads each from its
  source slot (source page * page size + offset) and writes them compactly into
  its own pages; one transfer segment per token, merged into a longer segment
  only where source and destination are both contiguous.  Section "Block RR
  改善哪一段": with whole blocks per rank, whole contiguous pages move.
"""

from __future__ import annotations

import numpy as np


class LayoutError(ValueError):
    """A position, page index or page id that the layout cannot place."""


def _check_layout(N: int, I: int, P: int | None = None) -> None:
    if N < 1 or I < 1:
        raise LayoutError(f"bad layout N={N} I={I}")
    if P is not None and (P < 1 or P % I != 0):
        # vLLM-Ascend "块表": block_size % cp_kv_cache_interleave_size == 0.
        raise LayoutError(f"page size {P} must be a positive multiple of interleave {I}")


def owner(p, N: int, I: int = 1):
    """Shard that stores position p: (p // I) % N (token RR when I == 1)."""
    _check_layout(N, I)
    p = np.asarray(p, dtype=np.int64)
    return (p // I) % N


def local_row(p, N: int, I: int = 1):
    """Compact local row of position p on its owner: (p // (N*I)) * I + p % I."""
    _check_layout(N, I)
    p = np.asarray(p, dtype=np.int64)
    return (p // (N * I)) * I + p % I


def global_pos(r, row, N: int, I: int = 1):
    """Inverse of (owner, local_row): position held by shard r at local row `row`.

    Local row rho of shard r is the (rho % I)-th token of the (rho // I)-th block
    that shard r received; blocks are dealt to shards in turn, so that block is
    global block (rho // I) * N + r.
    """
    _check_layout(N, I)
    row = np.asarray(row, dtype=np.int64)
    return (row // I) * (N * I) + np.int64(r) * I + row % I


def count(r, x, N: int, I: int = 1):
    """Number of positions p < x owned by shard r (the pages' local_len / count)."""
    _check_layout(N, I)
    x = np.asarray(x, dtype=np.int64)
    full = (x // (N * I)) * I
    rem = np.clip(x % (N * I) - np.int64(r) * I, 0, I)
    return full + rem


def chunk_share(r, a, L, N: int, I: int = 1):
    """Shard r's share of the chunk [a, a+L): count(a+L) - count(a)."""
    return count(r, np.asarray(a) + np.asarray(L), N, I) - count(r, a, N, I)


def physical_slot(block_table_row, row, P: int):
    """slot = page_id * P + offset_in_page for local row `row` (page = row // P)."""
    bt = np.asarray(block_table_row, dtype=np.int64)
    row = np.asarray(row, dtype=np.int64)
    page_idx = row // P
    if np.any(row < 0) or np.any(page_idx >= bt.shape[-1]):
        raise LayoutError("local row beyond the block table")
    return bt[..., page_idx] * P + row % P


def slot_map(pos, req, block_table, N: int, I: int, P: int):
    """(owner, local row, physical slot in the owner's pool) per new token."""
    _check_layout(N, I, P)
    pos = np.asarray(pos, dtype=np.int64)
    req = np.asarray(req, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    if np.any(pos < 0):
        raise LayoutError("negative position")
    own = owner(pos, N, I)
    row = local_row(pos, N, I)
    page_idx = row // P
    if np.any(page_idx >= bt.shape[1]):
        raise LayoutError("local row beyond the block table")
    slot = bt[req, page_idx] * P + row % P
    return own, row, slot


def vllm_slot(x, N: int, I: int, P: int, block_table_row):
    """vLLM-Ascend virtual-block mapping of request position x.

    Returns (rank, slot) with slot = block_table[x // vbs] * P + offset in the
    local block, following the formula of section "块表" step by step.
    """
    _check_layout(N, I, P)
    x = np.asarray(x, dtype=np.int64)
    bt = np.asarray(block_table_row, dtype=np.int64)
    vbs = P * N                       # virtual_block_size = block_size * cp_size
    vblock = x // vbs                 # (virtual) block index
    off = x % vbs                     # offset_within_virtual_block
    lbi = off // I                    # local_block_index
    rank = lbi % N                    # target_rank
    local_off = (lbi // N) * I + off % I
    return rank, bt[vblock] * P + local_off


def kv_append(arena, kv_new_bits, pos, req, block_table, N: int, I: int, P: int,
              shard_begin: int = 0, shard_end: int | None = None):
    """Owner-filtered write of latent rows into per-shard pools, in place.

    arena: uint16 (bf16 bit patterns) [shard_end - shard_begin, pool_pages * P, 576].
    Each new token's row is written only into its owner's pool, at the physical
    slot of its local row; tokens owned by shards outside [shard_begin, shard_end)
    are skipped ("MLA 的 Decode Context Parallelism", section 4 stage 2: every
    rank computes the latent, only the owner stores it).
    Raises LayoutError on a position, page index or page id out of range.
    """
    if shard_end is None:
        shard_end = N
    arena = np.asarray(arena)
    pool_rows = arena.shape[1]
    own, _row, slot = slot_map(pos, req, block_table, N, I, P)
    if np.any(slot < 0) or np.any(slot >= pool_rows):
        raise LayoutError("page id outside the pool")
    kv_new_bits = np.asarray(kv_new_bits)
    for t in range(len(own)):
        r = int(own[t])
        if shard_begin <= r < shard_end:
            arena[r - shard_begin, int(slot[t])] = kv_new_bits[t]
    return arena


def pd_relayout(arena, src_pool_bits, src_block_table, src_P: int, pos, req, block_table,
                N: int, I: int, P: int, shard_begin: int = 0, shard_end: int | None = None):
    """Prefill-to-decode relayout of latent rows, in place (section "PD + DCP").

    src_pool_bits: uint16 [src_rows, 576], the prefill side's paged pool (no
    context sharding); request b's position p lives at source row
    src_block_table[b][p // src_P] * src_P + p % src_P.  Each listed token
    (pos[t] of request req[t]) goes to its owner's pool at the slot dcp
    slot_map gives (owner by request position, compact local rows); tokens of
    shards outside [shard_begin, shard_end) are skipped.  Returns the arena and
    the (owner, source row, destination slot) of every token.
    Raises LayoutError on a position, page index or page id out of range.
    """
    if shard_end is None:
        shard_end = N
    pos = np.asarray(pos, dtype=np.int64)
    req = np.asarray(req, dtype=np.int64)
    src = np.asarray(src_pool_bits)
    # source side: one shard, pages of src_P rows (owner 0, local row = position)
    _o, _r, src_row = slot_map(pos, req, src_block_table, 1, 1, src_P)
    if np.any(src_row < 0) or np.any(src_row >= src.shape[0]):
        raise LayoutError("source page id outside the source pool")
    own, _row, dst = slot_map(pos, req, block_table, N, I, P)
    arena = np.asarray(arena)
    if np.any(dst < 0) or np.any(dst >= arena.shape[1]):
        raise LayoutError("page id outside the pool")
    for t in range(len(pos)):
        r = int(own[t])
        if shard_begin <= r < shard_end:
            arena[r - shard_begin, int(dst[t])] = src[int(src_row[t])]
    return arena, own, src_row, dst


def relayout_segments(src_rows, dst_slots):
    """Transfer segments (source row, destination slot, rows) of one rank's tokens.

    Tokens in request order, one segment each; consecutive tokens are merged
    only when both the source rows and the destination slots continue
    contiguously (section "PD + DCP").
    """
    segs = []
    for s_, d_ in zip(np.asarray(src_rows).tolist(), np.asarray(dst_slots).tolist()):
        if segs and segs[-1][0] + segs[-1][2] == s_ and segs[-1][1] + segs[-1][2] == d_:
            segs[-1][2] += 1
        else:
            segs.append([s_, d_, 1])
    return [tuple(x) for x in segs]


def accounting():
    """Byte counts the pages state for absorbed MLA (section 5 of the MLA page).

    Returns a dict computed from the K3 symbol table (d_c = 512, d_R = 64,
    H = 96, 24 MLA layers, d_model = 7168) and B = 64 at bf16.
    """
    d_c, d_r, H, layers, d_model, B, bf16 = 512, 64, 96, 24, 7168, 64, 2
    row = (d_c + d_r) * bf16
    return {
        "kv_bytes_per_token_layer": row,
        "kv_bytes_1m_24_layers": row * layers * 10**6,
        "q_allgather_bytes": B * H * (d_c + d_r) * bf16,
        "a2a_partial_bytes": B * H * (d_c + 4) * bf16,
        "o_proj_allreduce_bytes": B * d_model * bf16,
        "mha_kv_elems_per_token": 2 * H * 128,
        "mla_kv_elems_per_token": d_c + d_r,
    }
