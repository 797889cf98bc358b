"""The allocation-free partial decode (dcp_mla_decode_partial_static), through the C ABI.

That entry point serves callers that cannot allocate device memory for a
workspace (a serving process whose HBM is all given to its KV pool, or a plain
C host with no device-memory manager): it runs on a scratch array the library
owns.  These tests check that it gives the same partials as
dcp_mla_decode_partial with a caller workspace, on two calls in a row (the
second reuses whatever the first left in the shared scratch), that both match
the fp64 oracle, and that sizes beyond the array are rejected.  This file is
collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads

from harness import GpuState, assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu


def _static_call(st, o_part, lse_part, status):
    import context_sharded_mla_gb300 as dcp
    dcp.dcp_mla_decode_partial_static(st.layout, 0, st.cfg.N, st.q, st.dec.arena, st.pool_pages, st.bt,
                                      st.max_pages, st.seq_lens, workloads.SCALE, 1 if st.cfg.base == 2 else 0,
                                      o_part, lse_part, status)


@pytest.mark.parametrize("name,over", [("k3", dict(B=3, S=4096 + 13)),
                                       ("ragged", dict(B=5, S=3000, S_min=17))])
def test_static_scratch_matches_workspace_call(name, over):
    cfg = workloads.config(name, **over)
    st = GpuState(cfg, keep_kv=False)
    st.decode()                                     # reference: caller-provided workspace
    ref_o = to_f64(st.dec.o_part)
    ref_l = to_f64(st.dec.lse_part)
    # the oracle's per-shard partials of every request (fp64, from the same input rows)
    orc_o = np.zeros(ref_o.shape)
    orc_l = np.zeros(ref_l.shape)
    for b in range(cfg.B):
        _o, _l, o_parts, lse_parts = st.oracle_request(b)
        orc_o[:, b] = o_parts
        orc_l[:, b] = lse_parts
    for call in range(2):                           # two calls in a row share the scratch
        o_part = torch.full_like(st.dec.o_part, float("nan"))
        lse_part = torch.full_like(st.dec.lse_part, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _static_call(st, o_part, lse_part, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close_o(to_f64(o_part), ref_o, f"{name} static o_part call {call} vs workspace call")
        assert_close_lse(to_f64(lse_part), ref_l, f"{name} static lse_part call {call} vs workspace call")
        assert_close_o(to_f64(o_part), orc_o, f"{name} static o_part call {call} vs oracle")
        assert_close_lse(to_f64(lse_part), orc_l, f"{name} static lse_part call {call} vs oracle")


def test_static_scratch_rejects_oversized_request():
    import context_sharded_mla_gb300 as dcp
    lib = dcp.load_library()
    lay = dcp.Layout(8, 1, 64)
    cap = dcp.dcp_mla_decode_static_scratch_bytes()
    B = 2_000_000                                   # tile prefix sums alone exceed the array
    need = dcp.dcp_mla_decode_workspace_size(lay, 0, 8, B, 1, 96)
    assert need > cap
    P = ctypes.c_void_p(256)
    rc = lib.dcp_mla_decode_partial_static(ctypes.byref(lay), 0, 8, P, B, 1, 96, P, 1, P, 1, 1, P,
                                           ctypes.c_float(0.07), 0, P, 0, P, P, None)
    assert rc == dcp.DCP_ERR_TOO_LARGE
    assert lib.dcp_error_string(rc) == b"sizes need more scratch than the built-in area"
