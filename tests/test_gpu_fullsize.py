"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

Inputs are drawn on the GPU (seeded); the oracle recomputes sampled requests
(every head, or a head subset for the largest rows) in fp64 from the same
input rows, and checks the merged output and every shard's partial.  At least
64 (request, row) pairs per workload, each over the full sequence.
"""

import numpy as np
import pytest
import torch

import workloads

from harness import GpuState, assert_close_lse, assert_close_o, rel_row_err, to_f64

pytestmark = pytest.mark.gpu

SAMPLES = {
    "tiny": dict(reqs=[0], heads=None),
    "dsv3": dict(reqs=[0, 31], heads=None),
    "k3": dict(reqs=[0, 63], heads=None),
    "ragged": dict(reqs=None, heads=list(range(0, 128, 4))),
    "long": dict(reqs=[0], heads=None),
    "extend": dict(reqs=[3], heads=[0, 95]),
}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_fullsize_sampled(name):
    cfg = workloads.config(name)
    st = GpuState(cfg, gen_device="cuda", keep_kv=False)
    o, lse = st.decode()
    o = to_f64(o)
    lse = to_f64(lse)
    o_part = to_f64(st.dec.o_part)
    lse_part = to_f64(st.dec.lse_part)
    reqs = SAMPLES[name]["reqs"]
    if reqs is None:   # ragged: the shortest and the longest request
        S = st.S.numpy()
        reqs = [int(np.argmin(S)), int(np.argmax(S))]
    heads = SAMPLES[name]["heads"]
    hs = slice(None) if heads is None else heads
    worst = 0.0
    for b in reqs:
        ref_o, ref_lse, ref_op, ref_lp = st.oracle_request(b, heads)
        assert_close_o(o[b][:, hs], ref_o, f"{name} merged o b={b}")
        assert_close_lse(lse[b][:, hs], ref_lse, f"{name} merged lse b={b}")
        worst = max(worst, rel_row_err(o[b][:, hs], ref_o))
        for r in range(cfg.N):
            assert_close_o(o_part[r, b][:, hs], ref_op[r], f"{name} o_part r={r} b={b}")
            assert_close_lse(lse_part[r, b][:, hs], ref_lp[r], f"{name} lse_part r={r} b={b}")
    assert worst < 5e-2
    assert st.dec.status_bits() == 0
    # properties that hold at any size, on every row: finite outputs, lse finite
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    del st
    torch.cuda.empty_cache()
