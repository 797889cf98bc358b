"""Host-injected range errors on the decode call: the device status reports them,
no wait times out, and every other request is still exact.

The faults are bad inputs that the kernel range-checks before it reads
("PCP / DCP：计算、KV 布局与块轮转", section 9: validate the empty rank and the
tail block): a block-table page id outside the pool, and a max_pages too small
for one request's length.  Neither makes the GPU fault: the producer skips the
copy of that box and flags DCP_STATUS_BAD_PAGE_ID, and the partial of that
request is unspecified.
"""

import numpy as np
import pytest
import torch

import workloads

from harness import GpuState, assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu

BAD_PAGE_ID, TIMEOUT = 4, 32


def _decode(st, bt, max_pages):
    import context_sharded_mla_gb300 as dcp
    d = st.dec
    d.status.zero_()
    dcp.dcp_mla_decode_partial(d.layout, d.shard_begin, d.shard_end, st.q, d.arena, d.pool_pages, bt, max_pages,
                               st.seq_lens, d.scale, d.lse_base, d.o_part, d.lse_part, d.workspace, d.status)
    d.merge()
    torch.cuda.synchronize()
    return to_f64(d.o), to_f64(d.lse), to_f64(d.o_part), to_f64(d.lse_part), int(d.status.item())


def _check_others(st, o, lse, o_part, lse_part, bad_req):
    for b in range(st.cfg.B):
        if b == bad_req:
            continue
        ref_o, ref_lse, ref_op, ref_lp = st.oracle_request(b)
        assert_close_o(o[b], ref_o, f"merged o b={b}")
        assert_close_lse(lse[b], ref_lse, f"merged lse b={b}")
        for r in range(st.cfg.N):
            assert_close_o(o_part[r, b], ref_op[r], f"o_part r={r} b={b}")
            assert_close_lse(lse_part[r, b], ref_lp[r], f"lse_part r={r} b={b}")


@pytest.mark.parametrize("name,over,page", [
    ("k3", dict(B=4, S=4096 + 13), 3),            # pages of 64 rows: one TMA box per chunk and tile
    ("tiny", dict(B=3, S=1000), 5),               # pages of 16 rows: four boxes per tile
    ("ragged", dict(B=4, S=3000, S_min=400), 0),  # interleave 16, four query tokens
])
@pytest.mark.parametrize("bad_id", ["past_pool", "negative", "minus_two"])
def test_bad_page_id_in_one_request(name, over, page, bad_id):
    cfg = workloads.config(name, **over)
    st = GpuState(cfg)
    bad_req = 1
    bt = st.bt_cpu.clone()
    assert int(bt[bad_req, page]) >= 0                      # the entry is one the request uses
    bt[bad_req, page] = {"past_pool": st.pool_pages + 7, "negative": -3, "minus_two": -2}[bad_id]
    o, lse, o_part, lse_part, status = _decode(st, bt.to("cuda"), st.max_pages)
    assert status & BAD_PAGE_ID
    assert not status & TIMEOUT
    _check_others(st, o, lse, o_part, lse_part, bad_req)
    # the same state with the good table is exact everywhere (nothing was left behind)
    o, lse, o_part, lse_part, status = _decode(st, st.bt, st.max_pages)
    assert status == 0
    _check_others(st, o, lse, o_part, lse_part, None)


def test_max_pages_too_small_for_one_request():
    N, P = 8, 64
    S = (4096 + 13, 9000, 4096 + 13, 700)                   # 9, 18, 9 and 2 widened pages
    cfg = workloads.config("k3", B=len(S), lengths_override=S)
    st = GpuState(cfg)
    assert st.max_pages == 18
    o, lse, o_part, lse_part, status = _decode(st, st.bt, 9)  # request 1 needs 18
    assert status & BAD_PAGE_ID
    assert not status & TIMEOUT
    _check_others(st, o, lse, o_part, lse_part, 1)
