"""GPU parity of dcp_kv_relayout (prefill-to-decode relayout) against the oracle.

Rows are compared bit for bit (bf16 bit patterns): the pages' DCP1 -> DCP8
example for rank 1, the block-RR example, random chunks over several layouts
and shard subsets, bad entries (status bits, the other tokens still moved,
nothing else written), and a two-request 64K-token case.
"""

import json
import os

import numpy as np
import pytest
import torch

from oracle import layout as olayout

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENTINEL = -12345  # int16 pattern the pools start with


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def run_relayout(N, I, P, src_bits, src_bt, srcP, pos, req, bt, pool_pages, shard_begin=0, shard_end=None,
                 src_max_pages=None, max_pages=None):
    """GPU call; returns (arena bits [n, pool_rows, 576] int16 numpy, status)."""
    import context_sharded_mla_gb300 as dcp
    if shard_end is None:
        shard_end = N
    dev = "cuda"
    lay = dcp.Layout(N, I, P)
    src = torch.from_numpy(np.ascontiguousarray(src_bits)).view(torch.bfloat16).to(dev)
    arena = torch.full((shard_end - shard_begin, pool_pages * P, 576), SENTINEL, dtype=torch.int16,
                       device=dev).view(torch.bfloat16)
    sbt = torch.from_numpy(np.ascontiguousarray(src_bt, dtype=np.int32)).to(dev)
    dbt = torch.from_numpy(np.ascontiguousarray(bt, dtype=np.int32)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dcp.dcp_kv_relayout(lay, shard_begin, shard_end, src, srcP, sbt,
                        sbt.shape[1] if src_max_pages is None else src_max_pages,
                        torch.as_tensor(pos, dtype=torch.int64).to(dev), torch.as_tensor(req, dtype=torch.int32).to(dev),
                        dbt, dbt.shape[1] if max_pages is None else max_pages, arena, pool_pages, status)
    torch.cuda.synchronize()
    return arena.view(torch.int16).cpu().numpy(), int(status.item())


def oracle_arena(N, I, P, src_bits, src_bt, srcP, pos, req, bt, pool_pages, shard_begin=0, shard_end=None):
    if shard_end is None:
        shard_end = N
    arena = np.full((shard_end - shard_begin, pool_pages * P, 576), SENTINEL, dtype=np.int16)
    olayout.pd_relayout(arena, src_bits, src_bt, srcP, pos, req, bt, N, I, P, shard_begin, shard_end)
    return arena


def random_src(rows, seed):
    return np.random.default_rng(seed).integers(-32768, 32767, size=(rows, 576), dtype=np.int16)


def test_pages_dcp1_to_dcp8_example():
    g = golden("pd_relayout_rank1.json")
    N, r, P = g["N"], g["rank"], g["P"]
    pos = np.arange(g["request_tokens"])
    src = random_src(16 * P, 1)
    src_bt, bt = np.array([g["source_pages"]]), np.array([[g["dest_page"]]])
    got, st = run_relayout(N, 1, P, src, src_bt, P, pos, np.zeros_like(pos), bt, 11, r, r + 1)
    assert st == 0
    for s_, d_ in zip(g["source_slots"], g["dest_slots"]):
        assert np.array_equal(got[0, d_], src[s_])
    written = np.nonzero(np.any(got[0] != SENTINEL, axis=1))[0]
    assert list(written) == g["dest_slots"]
    want = oracle_arena(N, 1, P, src, src_bt, P, pos, np.zeros_like(pos), bt, 11, r, r + 1)
    assert np.array_equal(got, want)


def test_pages_block_rr_example():
    g = golden("pd_relayout_block_rr.json")
    N, Bk, P = g["N"], g["block"], g["P"]
    pos = np.arange(g["request_tokens"])
    src = random_src(16 * P, 2)
    src_bt, bt = np.array([g["source_pages"]]), np.array([[7]])
    got, st = run_relayout(N, Bk, P, src, src_bt, P, pos, np.zeros_like(pos), bt, 8)
    assert st == 0
    for k, r in enumerate(g["rank_of_block"]):
        sp = g["source_pages"][k]
        assert np.array_equal(got[r, 7 * P:8 * P], src[sp * P:(sp + 1) * P])
    assert np.all(got[3:] == SENTINEL)
    assert np.array_equal(got, oracle_arena(N, Bk, P, src, src_bt, P, pos, np.zeros_like(pos), bt, 8))


def make_case(N, I, P, srcP, B, L, starts, seed):
    rng = np.random.default_rng(seed)
    a = np.array(starts[:B])
    pos = np.concatenate([np.arange(a[b], a[b] + L) for b in range(B)])
    req = np.repeat(np.arange(B), L).astype(np.int32)
    src_pages = (a + L + srcP - 1) // srcP
    spmax = int(src_pages.max())
    src_bt = np.full((B, spmax), -1, dtype=np.int64)
    perm = rng.permutation(int(src_pages.sum()))
    k = 0
    for b in range(B):
        src_bt[b, :src_pages[b]] = perm[k:k + src_pages[b]]
        k += src_pages[b]
    rows = [int(olayout.count(0, a[b] + L, N, I)) + I for b in range(B)]
    dpages = max((x + P - 1) // P for x in rows)
    bt = rng.permutation(B * dpages).reshape(B, dpages)
    src = random_src(int(src_pages.sum()) * srcP, seed + 7)
    return src, src_bt, srcP, pos, req, bt, B * dpages


@pytest.mark.parametrize("N,I,P,srcP,sb,se", [(8, 1, 64, 64, 0, 8), (4, 2, 16, 32, 0, 4), (3, 5, 20, 16, 1, 3),
                                             (16, 16, 64, 128, 5, 11)])
def test_random_chunks_match_oracle(N, I, P, srcP, sb, se):
    src, src_bt, srcP, pos, req, bt, pool_pages = make_case(N, I, P, srcP, 3, 500, [0, 37, 1000], N * 10 + I)
    got, st = run_relayout(N, I, P, src, src_bt, srcP, pos, req, bt, pool_pages, sb, se)
    assert st == 0
    assert np.array_equal(got, oracle_arena(N, I, P, src, src_bt, srcP, pos, req, bt, pool_pages, sb, se))


def test_bad_entries_set_status_and_skip_only_those_tokens():
    N, I, P, srcP = 4, 1, 16, 16
    src, src_bt, srcP, pos, req, bt, pool_pages = make_case(N, I, P, srcP, 2, 200, [0, 5], 3)
    src_bt = src_bt.copy()
    src_bt[1, 2] = src.shape[0] // srcP          # a source page past the source pool
    pos = pos.copy()
    req = req.copy()
    pos[7] = -3                                   # a negative position
    req[11] = 9                                   # a request past B
    got, st = run_relayout(N, I, P, src, src_bt, srcP, pos, req, bt, pool_pages)
    assert st & 1 and st & 8 and st & 4
    bad = np.zeros(len(pos), dtype=bool)
    bad[7] = bad[11] = True
    bad |= (req == 1) & (pos // srcP == 2)
    ok = ~bad
    want = oracle_arena(N, I, P, src, src_bt, srcP, pos[ok], req[ok], bt, pool_pages)
    assert np.array_equal(got, want)


def test_two_long_requests():
    """Two 64K-token requests into 8 shards (token RR), whole arena compared."""
    N, I, P, srcP = 8, 1, 64, 64
    src, src_bt, srcP, pos, req, bt, pool_pages = make_case(N, I, P, srcP, 2, 65536, [0, 4096], 11)
    got, st = run_relayout(N, I, P, src, src_bt, srcP, pos, req, bt, pool_pages)
    assert st == 0
    own, _row, dst = olayout.slot_map(pos, req, bt, N, I, P)
    _o, _r, srow = olayout.slot_map(pos, req, src_bt, 1, 1, srcP)
    assert np.array_equal(got[own, dst], src[srow])
    assert int(np.sum(np.any(got != SENTINEL, axis=2))) == len(pos)   # nothing else written
