"""Pins for the oracle's slot mapping (no GPU).

Each test checks ``oracle.layout`` against something other than itself: the
worked examples printed on the pages (``tests/golden``), brute-force dealing of
positions (``oracle.bruteforce``), and invariants the layout must satisfy.
"""

import itertools
import json
import os

import numpy as np
import pytest

from oracle import bruteforce, layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_token_rr_example():
    g = golden("token_rr_n8.json")
    N, I = g["N"], g["I"]
    for r, positions in g["first_positions_per_rank"].items():
        p = np.array(positions)
        assert np.all(layout.owner(p, N, I) == int(r))
        # compact local storage: the k-th listed token is local row k
        assert list(layout.local_row(p, N, I)) == list(range(len(p)))


def test_block_rr_example():
    g = golden("block_rr_dcp4_b4.json")
    N, I = g["N"], g["I"]
    for lo, hi, r in g["owner_ranges"]:
        p = np.arange(lo, hi + 1)
        assert np.all(layout.owner(p, N, I) == r)
    for x, counts in g["counts_after"].items():
        got = [int(layout.count(r, int(x), N, I)) for r in range(N)]
        assert got == counts


def test_paged_slot_example():
    g = golden("paged_slots_p64.json")
    bt = np.array([g["pages"]])
    for lo, hi, slo, shi in g["ranges"]:
        p = np.arange(lo, hi + 1)
        own, row, slot = layout.slot_map(p, np.zeros_like(p), bt, g["N"], g["I"], g["P"])
        assert np.all(own == 0)
        assert list(slot) == list(range(slo, shi + 1))


def test_pd_relayout_example():
    """Owner filter on request positions + source slots + compact destination rows."""
    g = golden("pd_relayout_rank1.json")
    N, r, P = g["N"], g["rank"], g["P"]
    pos = np.arange(g["request_tokens"])
    mine = pos[layout.owner(pos, N, 1) == r]
    assert list(mine) == g["positions"]
    # source side is a non-DCP (N=1) request with pages [5, 9, 2]
    src_bt = np.array([g["source_pages"]])
    _, _, src_slot = layout.slot_map(mine, np.zeros_like(mine), src_bt, 1, 1, P)
    assert list(src_slot) == g["source_slots"]
    assert g["not_a_source_slot"] not in set(src_slot.tolist())
    # destination: rank r packs its tokens compactly into its own page 10
    dst_bt = np.array([[g["dest_page"]]])
    own, row, dst_slot = layout.slot_map(mine, np.zeros_like(mine), dst_bt, N, 1, P)
    assert np.all(own == r)
    assert list(dst_slot) == g["dest_slots"]
    assert len(mine) == g["tokens_received"] == int(layout.count(r, g["request_tokens"], N, 1))


LAYOUTS = [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (4, 4), (4, 2), (3, 5), (16, 16), (8, 3)]


@pytest.mark.parametrize("N,I", LAYOUTS)
def test_count_matches_dealing(N, I):
    X = 4 * N * I + 3
    lists = bruteforce.deal(X, N, I)
    for x in range(X + 1):
        dealt = bruteforce.deal(x, N, I)
        for r in range(N):
            assert int(layout.count(r, x, N, I)) == len(dealt[r])
    table = bruteforce.owner_row_table(X, N, I)
    p = np.arange(X)
    own = layout.owner(p, N, I)
    row = layout.local_row(p, N, I)
    for i in range(X):
        assert (int(own[i]), int(row[i])) == table[i]
    for r in range(N):
        rows = np.arange(len(lists[r]))
        assert list(layout.global_pos(r, rows, N, I)) == lists[r]


@pytest.mark.parametrize("N,I", LAYOUTS)
def test_bijection_and_balance(N, I):
    for S in list(range(0, 3 * N * I + 2)) + [1000, 4097]:
        p = np.arange(S)
        own = layout.owner(p, N, I)
        row = layout.local_row(p, N, I)
        counts = np.array([int(layout.count(r, S, N, I)) for r in range(N)])
        assert counts.sum() == S
        for r in range(N):
            rows_r = np.sort(row[own == r])
            # shard r holds exactly local rows 0 .. count_r(S)-1, each once
            assert list(rows_r) == list(range(counts[r]))
        # balance: token RR within one token; block RR within I tokens
        assert counts.max() - counts.min() <= (1 if I == 1 else I)
        pairs = set(zip(own.tolist(), row.tolist()))
        assert len(pairs) == S


@pytest.mark.parametrize("N,I", LAYOUTS)
def test_chunk_share(N, I):
    rng = np.random.default_rng(N * 100 + I)
    for _ in range(50):
        a = int(rng.integers(0, 5 * N * I))
        L = int(rng.integers(0, 7 * N * I))
        shares = [int(layout.chunk_share(r, a, L, N, I)) for r in range(N)]
        assert sum(shares) == L
        p = np.arange(a, a + L)
        for r in range(N):
            assert shares[r] == int(np.sum(layout.owner(p, N, I) == r))


@pytest.mark.parametrize("N,I,P", [(8, 1, 64), (4, 4, 16), (16, 16, 64), (2, 2, 8), (3, 1, 5), (8, 8, 64), (4, 2, 6)])
def test_vllm_virtual_block_equals_block_rr(N, I, P):
    """vLLM-Ascend's virtual-block slot equals the shared-block-table slot when I | P."""
    rng = np.random.default_rng(7)
    pages = 12
    bt = rng.permutation(100)[:pages]
    x = np.arange(pages * N * P)
    rank_v, slot_v = layout.vllm_slot(x, N, I, P, bt)
    own, _row, slot = layout.slot_map(x, np.zeros_like(x), bt[None, :], N, I, P)
    assert np.array_equal(rank_v, own)
    assert np.array_equal(slot_v, slot)


def test_interleave_must_divide_page():
    with pytest.raises(layout.LayoutError):
        layout.slot_map([0], [0], [[0]], 4, 3, 16)


def test_slot_range_errors():
    bt = np.array([[3, 1]])
    with pytest.raises(layout.LayoutError):
        layout.slot_map([4 * 2 * 4], [0], bt, 4, 1, 4)    # local row 8 -> page index 2
    with pytest.raises(layout.LayoutError):
        layout.slot_map([-1], [0], bt, 4, 1, 4)


def test_kv_append_owner_filtered():
    N, I, P = 4, 2, 4
    S = 29
    bt = np.array([[2, 0, 3, 1]])
    pool_pages = 4
    rng = np.random.default_rng(3)
    kv = rng.integers(0, 65535, size=(S, 576), dtype=np.uint16)
    arena = np.zeros((N, pool_pages * P, 576), np.uint16)
    pos = np.arange(S)
    layout.kv_append(arena, kv, pos, np.zeros_like(pos), bt, N, I, P)
    for r in range(N):
        n = int(layout.count(r, S, N, I))
        for rho in range(n):
            p = int(layout.global_pos(r, rho, N, I))
            s = int(bt[0, rho // P]) * P + rho % P
            assert np.array_equal(arena[r, s], kv[p])
    # shard-range filter: only shards [1, 3) are held; others are skipped
    sub = np.zeros((2, pool_pages * P, 576), np.uint16)
    layout.kv_append(sub, kv, pos, np.zeros_like(pos), bt, N, I, P, 1, 3)
    assert np.array_equal(sub, arena[1:3])
    # an out-of-pool page id is an error
    bad = np.array([[2, 9, 3, 1]])
    with pytest.raises(layout.LayoutError):
        layout.kv_append(arena, kv, pos, np.zeros_like(pos), bad, N, I, P)


def test_accounting_matches_pages():
    g = golden("mla_accounting.json")
    a = layout.accounting()
    assert a["kv_bytes_per_token_layer"] == 1152
    assert abs(a["kv_bytes_per_token_layer"] / 1024 - g["kv_bytes_per_token_layer"]["approx_KB"]) < 1e-9
    assert abs(a["kv_bytes_1m_24_layers"] / 1e9 - g["kv_1m_24_layers"]["approx_GB"]) < 0.05
    assert abs(a["kv_bytes_1m_24_layers"] / 8 / 1e9 - g["per_rank_cp8_GB"]) < 0.01
    assert abs(a["q_allgather_bytes"] / 1e6 - g["q_allgather"]["approx_MB"]) < 0.05
    assert abs(a["q_allgather_bytes"] * 7 / 8 / 1e6 - g["q_allgather"]["sent_per_rank_MB"]) < 0.05
    assert abs(a["a2a_partial_bytes"] / 1e6 - g["a2a_partials"]["approx_MB"]) < 0.05
    assert abs(a["a2a_partial_bytes"] * 7 / 8 / 1e6 - g["a2a_partials"]["sent_per_rank_MB"]) < 0.05
    assert abs(a["o_proj_allreduce_bytes"] / 1e6 - g["o_proj_allreduce"]["approx_MB"]) < 0.005
    assert abs(a["o_proj_allreduce_bytes"] * 2 * 7 / 8 / 1e6 - g["o_proj_allreduce"]["ring_per_rank_MB"]) < 0.05
    assert a["mha_kv_elems_per_token"] == g["mha_per_token"]["value"]
    assert round(a["mha_kv_elems_per_token"] / a["mla_kv_elems_per_token"]) == 43


def test_layout_exhaustive_small():
    """Every (N, I) with N, I <= 5: owner/row from formulas equal dealing for S <= 60."""
    for N, I in itertools.product(range(1, 6), range(1, 6)):
        table = bruteforce.owner_row_table(60, N, I)
        p = np.arange(60)
        own = layout.owner(p, N, I)
        row = layout.local_row(p, N, I)
        assert all((int(own[i]), int(row[i])) == table[i] for i in range(60))


def _src_pool(rows):
    """A source pool whose row k holds the bit pattern k in every dim (uint16)."""
    return np.repeat(np.arange(rows, dtype=np.uint16)[:, None], 576, axis=1)


def test_pd_relayout_copies_the_worked_example():
    """The owner-filtered copy moves exactly the page's 24 tokens, one segment each."""
    g = golden("pd_relayout_rank1.json")
    N, r, P = g["N"], g["rank"], g["P"]
    pos = np.arange(g["request_tokens"])
    src = _src_pool(16 * P)
    arena = np.full((1, 16 * P, 576), 0xFFFF, dtype=np.uint16)
    arena, own, src_row, dst = layout.pd_relayout(arena, src, np.array([g["source_pages"]]), P, pos,
                                                  np.zeros_like(pos), np.array([[g["dest_page"]]]), N, 1, P,
                                                  shard_begin=r, shard_end=r + 1)
    mine = own == r
    assert list(src_row[mine]) == g["source_slots"]
    assert list(dst[mine]) == g["dest_slots"]
    for s_, d_ in zip(g["source_slots"], g["dest_slots"]):
        assert np.all(arena[0, d_] == s_)
    written = np.nonzero(np.any(arena[0] != 0xFFFF, axis=1))[0]
    assert list(written) == g["dest_slots"]          # nothing else in rank 1's pool changed
    segs = layout.relayout_segments(src_row[mine], dst[mine])
    assert len(segs) == g["tokens_received"] and all(n == 1 for _, _, n in segs)


def test_pd_relayout_block_rr_moves_whole_pages():
    """Block RR: request block k goes whole to rank k % N, as one contiguous segment."""
    g = golden("pd_relayout_block_rr.json")
    N, Bk, P = g["N"], g["block"], g["P"]
    pos = np.arange(g["request_tokens"])
    dst_page = 7
    arena = np.zeros((N, 8 * P, 576), dtype=np.uint16)
    arena, own, src_row, dst = layout.pd_relayout(arena, _src_pool(16 * P), np.array([g["source_pages"]]), P, pos,
                                                  np.zeros_like(pos), np.array([[dst_page]]), N, Bk, P)
    for k, r in enumerate(g["rank_of_block"]):
        blk = own[k * Bk:(k + 1) * Bk]
        assert np.all(blk == r)
        segs = layout.relayout_segments(src_row[own == r], dst[own == r])
        assert segs == [(g["source_pages"][k] * P, dst_page * P, Bk)]
    assert [int(np.sum(own == r)) for r in range(N)] == g["rows_per_rank"]


@pytest.mark.parametrize("N,I,P,srcP", [(8, 1, 64, 64), (4, 2, 16, 32), (3, 5, 20, 16), (16, 16, 64, 128)])
def test_pd_relayout_matches_brute_force(N, I, P, srcP):
    """Every token lands once, in its owner's pool at the dealt local row; chunk shares match count()."""
    rng = np.random.default_rng(N * 100 + I)
    B, L = 3, 300
    a = np.array([0, 37, 1000])                       # chunk start of each request
    pos = np.concatenate([np.arange(a[b], a[b] + L) for b in range(B)])
    req = np.repeat(np.arange(B), L)
    src_pages = (a + L + srcP - 1) // srcP
    src_bt = np.full((B, int(src_pages.max())), -1, dtype=np.int64)
    perm = rng.permutation(int(src_pages.sum()))
    k = 0
    for b in range(B):
        src_bt[b, :src_pages[b]] = perm[k:k + src_pages[b]]
        k += src_pages[b]
    rows_per_b = [int(layout.count(0, a[b] + L, N, I)) + I for b in range(B)]
    dpages = max((r + P - 1) // P for r in rows_per_b)
    bt = rng.permutation(B * dpages).reshape(B, dpages)
    src = rng.integers(0, 65535, size=(int(src_pages.sum()) * srcP, 576), dtype=np.uint16)
    arena = np.zeros((N, B * dpages * P, 576), dtype=np.uint16)
    arena, own, src_row, dst = layout.pd_relayout(arena, src, src_bt, srcP, pos, req, bt, N, I, P)
    dealt = bruteforce.owner_row_table(int(a.max()) + L, N, I)
    for t in range(len(pos)):
        b, p = int(req[t]), int(pos[t])
        r, rho = dealt[p]
        assert own[t] == r
        assert src_row[t] == src_bt[b, p // srcP] * srcP + p % srcP
        assert dst[t] == bt[b, rho // P] * P + rho % P
        assert np.array_equal(arena[r, dst[t]], src[src_row[t]])
    for b in range(B):
        for r in range(N):
            got = int(np.sum((req == b) & (own == r)))
            assert got == int(layout.count(r, a[b] + L, N, I) - layout.count(r, a[b], N, I))
