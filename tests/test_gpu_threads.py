"""Two host threads driving the library on one GPU at once, against the fp64 oracle.

The library's host state (the raised shared-memory limit of each kernel, the
occupancy figure the partial decode plans with, the tensor-map encoder) is
per device and guarded by locks, so that one host thread per GPU, or several
threads on one GPU with their own streams and buffers, may call every entry
point at the same time.  ctypes drops the GIL for the length of each call, so
the two threads below are inside the library together.  Each thread appends
its own workload, then decodes it several times on its own stream; every
result is compared with the oracle.
"""

import threading

import numpy as np
import pytest
import torch

import workloads

from harness import GpuState, assert_close_lse, assert_close_o, to_f64

pytestmark = pytest.mark.gpu

REPEATS = 4


def _worker(name, over, start, out, errors):
    try:
        cfg = workloads.config(name, **over)
        stream = torch.cuda.Stream()
        start.wait(timeout=60)
        with torch.cuda.stream(stream):
            st = GpuState(cfg, keep_kv=True)          # append through the library on this stream
            results = []
            for _ in range(REPEATS):
                o, lse = st.dec.decode(st.q, st.bt, st.seq_lens, stream)
                results.append((o.clone(), lse.clone()))
        stream.synchronize()
        out[name] = (st, results)
    except Exception as e:  # reported by the main thread
        errors.append((name, repr(e)))


def test_two_threads_decode_concurrently():
    cases = [("k3", dict(B=3, S=3000 + 7, seed=21)), ("ragged", dict(B=4, S=2500, S_min=33, seed=22))]
    start = threading.Barrier(len(cases))
    out, errors = {}, []
    threads = [threading.Thread(target=_worker, args=(n, o, start, out, errors)) for n, o in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    for name, _over in cases:
        st, results = out[name]
        assert st.dec.status_bits() == 0
        for b in range(st.cfg.B):
            o_ref, l_ref, _op, _lp = st.oracle_request(b)
            for i, (o, lse) in enumerate(results):
                assert_close_o(to_f64(o[b]), o_ref, f"{name} thread call {i} b={b}")
                assert_close_lse(to_f64(lse[b]), l_ref, f"{name} thread call {i} b={b}")
        first = to_f64(results[0][0])
        for o, _lse in results[1:]:
            assert np.array_equal(to_f64(o), first), f"{name}: repeated decodes differ"
