"""GPU parity of the integer/copy steps: dcp_slot_map and dcp_kv_append (bit-exact)."""

import numpy as np
import pytest
import torch

import workloads
from oracle import layout as olayout

from harness import bits

pytestmark = pytest.mark.gpu


def _lib():
    import context_sharded_mla_gb300 as dcp
    dcp.load_library()
    return dcp


@pytest.mark.parametrize("N,I,P", [(4, 1, 16), (8, 1, 64), (16, 16, 64), (4, 4, 8), (3, 1, 5), (1, 1, 64)])
def test_slot_map_bit_exact(N, I, P):
    dcp = _lib()
    rng = np.random.default_rng(N * 7 + I)
    B = 5
    S = rng.integers(1, 3 * N * P + 17, size=B)
    cfg = workloads.config("tiny", B=B, N=N, I=I, P=P, lengths_override=tuple(int(s) for s in S))
    bt, pool_pages = workloads.block_table(cfg, torch.tensor(S))
    pos = np.concatenate([np.arange(s) for s in S]).astype(np.int64)
    req = np.concatenate([np.full(s, b) for b, s in enumerate(S)]).astype(np.int32)
    T = len(pos)
    dev = "cuda"
    owner = torch.empty(T, dtype=torch.int32, device=dev)
    row = torch.empty(T, dtype=torch.int64, device=dev)
    slot = torch.empty(T, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lay = dcp.Layout(N, I, P)
    dcp.dcp_slot_map(lay, torch.from_numpy(pos).to(dev), torch.from_numpy(req).to(dev), bt.to(dev),
                     bt.shape[1], pool_pages, owner, row, slot, status)
    torch.cuda.synchronize()
    o_own, o_row, o_slot = olayout.slot_map(pos, req, bt.numpy(), N, I, P)
    assert int(status.item()) == 0
    assert np.array_equal(owner.cpu().numpy(), o_own)
    assert np.array_equal(row.cpu().numpy(), o_row)
    assert np.array_equal(slot.cpu().numpy(), o_slot)
    # chunk shares from the host ABI equal the oracle's count differences
    for r in range(N):
        for a, L in [(0, 100), (37, 8192), (1000, 1)]:
            got = dcp.dcp_count(lay, r, a + L) - dcp.dcp_count(lay, r, a)
            assert got == int(olayout.chunk_share(r, a, L, N, I))


def test_slot_map_range_errors_set_status():
    dcp = _lib()
    dev = "cuda"
    lay = dcp.Layout(4, 1, 4)
    bt = torch.tensor([[3, 1], [0, 7]], dtype=torch.int32, device=dev)   # page 7 is outside a 4-page pool
    pos = torch.tensor([0, -5, 4 * 4 * 2, 20, 5], dtype=torch.int64, device=dev)
    req = torch.tensor([0, 0, 0, 1, 9], dtype=torch.int32, device=dev)
    T = 5
    owner = torch.empty(T, dtype=torch.int32, device=dev)
    row = torch.empty(T, dtype=torch.int64, device=dev)
    slot = torch.empty(T, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dcp.dcp_slot_map(lay, pos, req, bt, 2, 4, owner, row, slot, status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & 1 and st & 2 and st & 4 and st & 8
    s = slot.cpu().tolist()
    assert s[0] == 3 * 4 + 0 and s[1] == -1 and s[2] == -1 and s[3] == -1 and s[4] == -1


@pytest.mark.parametrize("name,N,I,P", [("tiny", 4, 1, 16), ("ragged", 16, 16, 64), ("k3", 8, 1, 64)])
def test_kv_append_bit_exact(name, N, I, P):
    dcp = _lib()
    B = 3
    S = (N * P * 2 + 5, 7, N * I + 1)
    cfg = workloads.config(name, B=B, N=N, I=I, P=P, lengths_override=S, H=4, q_len=1)
    bt, pool_pages = workloads.block_table(cfg, torch.tensor(S))
    dev = "cuda"
    lay = dcp.Layout(N, I, P)
    arena = torch.zeros(N, pool_pages * P, 576, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ref = np.zeros((N, pool_pages * P, 576), np.uint16)
    btd = bt.to(dev)
    for b in range(B):
        kv = workloads.gen_kv(cfg, b, S[b])
        pos = np.arange(S[b], dtype=np.int64)
        req = np.full(S[b], b, np.int32)
        dcp.dcp_kv_append(lay, 0, N, kv.to(dev), torch.from_numpy(pos).to(dev), torch.from_numpy(req).to(dev),
                          btd, bt.shape[1], arena, pool_pages, status)
        olayout.kv_append(ref, bits(kv), pos, req, bt.numpy(), N, I, P)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(arena), ref)
    # shard-range filter: a device holding shards [1, 3) writes only those pools
    sub = torch.zeros(2, pool_pages * P, 576, dtype=torch.bfloat16, device=dev)
    kv = workloads.gen_kv(cfg, 0, S[0])
    pos = np.arange(S[0], dtype=np.int64)
    dcp.dcp_kv_append(lay, 1, 3, kv.to(dev), torch.from_numpy(pos).to(dev),
                      torch.zeros(S[0], dtype=torch.int32, device=dev), btd, bt.shape[1], sub, pool_pages, status)
    ref_sub = np.zeros((2, pool_pages * P, 576), np.uint16)
    olayout.kv_append(ref_sub, bits(kv), pos, np.zeros(S[0], np.int32), bt.numpy(), N, I, P, 1, 3)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(sub), ref_sub)


def test_kv_append_mixed_requests_one_call():
    """One call with the tokens of every request in shuffled order (a decode step's batch)."""
    dcp = _lib()
    N, I, P, B = 8, 1, 64, 5
    S = (3 * N * P + 11, 1, 600, N + 2, 64 * N)
    cfg = workloads.config("k3", B=B, N=N, I=I, P=P, lengths_override=S, H=4, q_len=1)
    bt, pool_pages = workloads.block_table(cfg, torch.tensor(S))
    rng = np.random.default_rng(11)
    pos = np.concatenate([np.arange(s, dtype=np.int64) for s in S])
    req = np.concatenate([np.full(s, b, np.int32) for b, s in enumerate(S)])
    perm = rng.permutation(pos.size)
    pos, req = pos[perm], req[perm]
    kv = torch.from_numpy(rng.integers(0, 1 << 16, size=(pos.size, 576), dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)
    dev = "cuda"
    arena = torch.zeros(N, pool_pages * P, 576, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dcp.dcp_kv_append(dcp.Layout(N, I, P), 0, N, kv.to(dev), torch.from_numpy(pos).to(dev),
                      torch.from_numpy(req).to(dev), bt.to(dev), bt.shape[1], arena, pool_pages, status)
    ref = np.zeros((N, pool_pages * P, 576), np.uint16)
    olayout.kv_append(ref, bits(kv), pos, req, bt.numpy(), N, I, P)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(arena), ref)


def test_kv_append_range_errors_set_status():
    """Bad tokens set their status bit and are skipped; every other token is still written."""
    dcp = _lib()
    dev = "cuda"
    N, I, P = 2, 1, 4
    lay = dcp.Layout(N, I, P)
    bt = torch.tensor([[3, 9], [1, 0]], dtype=torch.int32)  # page 9 is outside a 4-page pool
    pool_pages = 4
    # token: good (b0, p0) | negative position | request 2 of 2 | local row 8 -> page index 2 of max 2
    #        | b0 p8 -> local row 4 -> page 9 (bad id) | good (b1, p3)
    pos = np.array([0, -1, 1, 16, 8, 3], np.int64)
    req = np.array([0, 0, 2, 1, 0, 1], np.int32)
    kv = torch.arange(6 * 576, dtype=torch.float32).reshape(6, 576).to(torch.bfloat16)
    arena = torch.zeros(N, pool_pages * P, 576, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dcp.dcp_kv_append(lay, 0, N, kv.to(dev), torch.from_numpy(pos).to(dev), torch.from_numpy(req).to(dev),
                      bt.to(dev), 2, arena, pool_pages, status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 1 | 2 | 4 | 8
    ref = np.zeros((N, pool_pages * P, 576), np.uint16)
    good = [0, 5]
    olayout.kv_append(ref, bits(kv)[good], pos[good], req[good], bt.numpy(), N, I, P)
    assert np.array_equal(bits(arena), ref)
