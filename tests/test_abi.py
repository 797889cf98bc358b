"""The C-ABI library builds, loads and exports every symbol include/dcp.h declares (no GPU).

Also checks the host-only parts: dcp_count against the oracle, and that bad
arguments are rejected on the host before anything is launched.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import layout as olayout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from context_sharded_mla_gb300 import _build, load_library
    _build.build()
    return load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dcp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dcp_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["dcp_count", "dcp_slot_map", "dcp_kv_append", "dcp_mla_decode_partial",
              "dcp_mla_decode_workspace_size", "dcp_lse_merge", "dcp_kv_relayout", "dcp_absorb_q",
              "dcp_absorb_o"]:
        assert n in names


def declared_parameters():
    """{function name: [parameter declarations]} from include/dcp.h."""
    src = open(os.path.join(ROOT, "include", "dcp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(dcp_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = params
    return out


# The calls the boundary specification lists, with its argument count, and every
# argument this library adds, with why (the departures are stated in the design
# notes as readings).
BOUNDARY = {
    "dcp_count": (3, []),
    "dcp_slot_map": (12, ["B", "pool_pages"]),                   # range checks of req and of page ids
    "dcp_kv_append": (12, ["shard_begin", "shard_end", "B"]),    # pools held by this device; req range check
    "dcp_mla_decode_partial": (22, []),
    "dcp_mla_decode_workspace_size": (5, ["shard_begin", "shard_end", "-max_seq"]),  # units depend on shards held,
                                                                                     # not on any length
    "dcp_lse_merge": (10, []),
}


def test_boundary_argument_counts():
    params = declared_parameters()
    for name, (spec_count, changes) in BOUNDARY.items():
        assert name in params, name
        added = sum(1 for c in changes if not c.startswith("-"))
        removed = sum(1 for c in changes if c.startswith("-"))
        assert len(params[name]) == spec_count + added - removed, (name, params[name])
        names = [p.split()[-1].lstrip("*") for p in params[name]]
        for c in changes:
            if c.startswith("-"):
                assert c[1:] not in names, (name, c)
            else:
                assert c in names, (name, c)


def test_binding_signatures_match_the_header():
    import context_sharded_mla_gb300 as dcp
    params = declared_parameters()
    for name, (_res, args) in dcp._SIGNATURES.items():
        assert name in params, f"{name} bound but not declared"
        assert len(args) == len(params[name]), (name, len(args), params[name])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/dcp.h but not exported"


def test_version_and_errors(lib):
    assert lib.dcp_version() >= 10000
    assert lib.dcp_error_string(-1) == b"invalid argument"
    assert lib.dcp_error_string(0) == b"ok"


@pytest.mark.parametrize("N,I", [(1, 1), (4, 1), (8, 1), (16, 16), (4, 4), (3, 2)])
def test_dcp_count_matches_oracle(lib, N, I):
    from context_sharded_mla_gb300 import Layout, dcp_count
    lay = Layout(N, I, I * 4)
    for r in range(N):
        for x in list(range(0, 5 * N * I)) + [10**6 + 3, 2**40 + 17]:
            assert dcp_count(lay, r, x) == int(olayout.count(r, x, N, I))


def test_host_validation_rejects_bad_arguments(lib):
    from context_sharded_mla_gb300 import Layout
    bad = Layout(4, 3, 16)          # interleave does not divide the page
    good = Layout(4, 1, 16)
    P = ctypes.c_void_p
    assert lib.dcp_count(ctypes.byref(bad), 0, 5) == -1
    assert lib.dcp_count(ctypes.byref(good), 4, 5) == -1
    assert lib.dcp_count(ctypes.byref(good), 0, -1) == -1
    assert lib.dcp_slot_map(ctypes.byref(bad), P(16), P(16), 1, P(16), 1, 1, 1, 1, P(16), P(16), P(16),
                            P(16), None) == -1
    assert lib.dcp_slot_map(ctypes.byref(good), P(16), P(16), 0, P(16), 1, 1, 1, 1, P(16), P(16), P(16),
                            P(16), None) == 0       # T == 0 is a no-op
    # append: (layout, shard_begin, shard_end, kv_new, pos, req, T, block_table, B, bt_stride, max_pages,
    #          arena, pool_pages, status, stream)
    ap = lambda **kw: dict(dict(sb=0, se=4, kv=P(16), pos=P(16), req=P(16), T=1, bt=P(16), B=1, st=1, mp=1,
                                ar=P(16), pp=1, status=P(16)), **kw)

    def append(**kw):
        a = ap(**kw)
        return lib.dcp_kv_append(ctypes.byref(good), a["sb"], a["se"], a["kv"], a["pos"], a["req"], a["T"], a["bt"],
                                 a["B"], a["st"], a["mp"], a["ar"], a["pp"], a["status"], None)
    assert append(T=0) == 0                         # no-op, nothing launched
    assert append(se=5) == -1
    assert append(kv=P(17)) == -1                   # not 16-byte aligned
    assert append(B=0) == -1
    assert append(mp=2, st=1) == -1
    assert append(pp=0) == -1
    assert append(pos=None) == -1
    assert lib.dcp_kv_append(ctypes.byref(bad), 0, 4, P(16), P(16), P(16), 1, P(16), 1, 1, 1, P(16), 1, P(16),
                             None) == -1
    # decode: q_len*H over the limit, bad base, bad dtype, missing workspace
    args = lambda **kw: dict(dict(sb=0, se=4, q=P(256), B=1, ql=1, H=16, ar=P(256), pp=1, bt=P(256), st=1, mp=1,
                                  sl=P(256), sc=0.1, base=0, op=P(256), od=0, lp=P(256), ws=None, wsb=0,
                                  status=P(256)), **kw)

    def call(**kw):
        a = args(**kw)
        return lib.dcp_mla_decode_partial(ctypes.byref(good), a["sb"], a["se"], a["q"], a["B"], a["ql"], a["H"],
                                          a["ar"], a["pp"], a["bt"], a["st"], a["mp"], a["sl"], a["sc"], a["base"],
                                          a["op"], a["od"], a["lp"], a["ws"], a["wsb"], a["status"], None)
    assert call(H=65537) == -1                      # more than 65536 query rows per request
    assert call(ql=512, H=129) == -1
    assert call(base=7) == -1
    assert call(od=9) == -1
    assert call(sc=-1.0) == -1
    assert call(se=5) == -1
    assert call(q=None) == -1
    assert call(mp=2, st=1) == -1
    # the allocation-free variant checks its arguments the same way, before any CUDA call

    def call_static(**kw):
        a = args(**kw)
        return lib.dcp_mla_decode_partial_static(ctypes.byref(good), a["sb"], a["se"], a["q"], a["B"], a["ql"],
                                                 a["H"], a["ar"], a["pp"], a["bt"], a["st"], a["mp"], a["sl"],
                                                 a["sc"], a["base"], a["op"], a["od"], a["lp"], a["status"], None)
    for bad_arg in (dict(H=65537), dict(base=7), dict(od=9), dict(sc=-1.0), dict(se=5), dict(q=None),
                    dict(mp=2, st=1), dict(q=P(264))):
        assert call_static(**bad_arg) == -1, bad_arg
    need = lib.dcp_mla_decode_workspace_size(ctypes.byref(good), 0, 4, 1, 1, 16)
    if need > 0:
        assert call(wsb=need - 1, ws=P(256)) == -4
    # prefill-to-decode relayout
    rl = lambda **kw: dict(dict(sb=0, se=4, src=P(256), srows=64, sps=16, sbt=P(256), sst=1, smp=1, pos=P(256),
                                req=P(256), T=1, B=1, bt=P(256), st=1, mp=1, ar=P(256), pp=1, status=P(256)), **kw)

    def relayout(**kw):
        a = rl(**kw)
        return lib.dcp_kv_relayout(ctypes.byref(good), a["sb"], a["se"], a["src"], a["srows"], a["sps"], a["sbt"],
                                   a["sst"], a["smp"], a["pos"], a["req"], a["T"], a["B"], a["bt"], a["st"],
                                   a["mp"], a["ar"], a["pp"], a["status"], None)
    assert relayout(T=0) == 0                       # no-op, nothing launched
    assert relayout(se=5) == -1
    assert relayout(sb=2, se=2) == -1
    assert relayout(sps=0) == -1
    assert relayout(smp=2, sst=1) == -1
    assert relayout(mp=0) == -1
    assert relayout(B=0) == -1
    assert relayout(src=P(264)) == -1               # not 16-byte aligned
    assert relayout(src=None) == -1
    assert relayout(status=None) == -1
    assert lib.dcp_kv_relayout(ctypes.byref(bad), 0, 4, P(256), 64, 16, P(256), 1, 1, P(256), P(256), 1, 1, P(256),
                               1, 1, P(256), 1, P(256), None) == -1
    # merge
    assert lib.dcp_lse_merge(0, 10, P(256), 0, P(256), 0, P(256), 0, P(256), None) == -1
    assert lib.dcp_lse_merge(2, 10, P(256), 3, P(256), 0, P(256), 0, P(256), None) == -1
    assert lib.dcp_lse_merge(2, 0, None, 0, None, 0, None, 0, None, None) == 0
    # absorption products
    aq = lambda **kw: dict(dict(T=4, H=8, qn=P(256), sn=192, qp=P(512), sp=192, w=P(1024), q=P(2048)), **kw)

    def absorb_q(**kw):
        a = aq(**kw)
        return lib.dcp_absorb_q(a["T"], a["H"], a["qn"], a["sn"], a["qp"], a["sp"], a["w"], a["q"], None, None)
    assert absorb_q(T=0) == 0                       # no-op, nothing launched
    assert absorb_q(T=-1) == -1
    assert absorb_q(H=0) == -1
    assert absorb_q(H=70000) == -1
    assert absorb_q(T=128 * 65536) == -1            # more token tiles than a grid dimension holds
    assert absorb_q(sn=100) == -1                   # shorter than the 128 dims read
    assert absorb_q(sn=196) == -1                   # not a multiple of 8 elements
    assert absorb_q(sp=60) == -1
    assert absorb_q(qn=P(264)) == -1                # not 16-byte aligned
    assert absorb_q(w=None) == -1
    assert absorb_q(q=None) == -1

    def absorb_o(T=4, H=8, o=P(256), od=0, w=P(512), v=P(1024), vd=1):
        return lib.dcp_absorb_o(T, H, o, od, w, v, vd, None, None)
    assert absorb_o(T=0) == 0
    assert absorb_o(od=2) == -1
    assert absorb_o(vd=-1) == -1
    assert absorb_o(T=0, od=5) == -1                # dtypes are checked even for an empty call
    assert absorb_o(o=None) == -1
    assert absorb_o(v=P(1032)) == -1
    assert absorb_o(H=0) == -1
    # the merge and the output product in one call

    def merge_absorb(n=8, T=4, H=8, o=P(256), od=0, lp=P(256), base=1, w=P(512), v=P(1024), vd=1):
        return lib.dcp_lse_merge_absorb_o(n, T, H, o, od, lp, base, w, v, vd, None, None, None)
    assert merge_absorb(T=0) == 0                   # no-op, nothing launched
    assert merge_absorb(n=0) == -1
    assert merge_absorb(n=65) == -1                 # more parts than the kernel's weight buffers hold
    assert merge_absorb(T=-1) == -1
    assert merge_absorb(H=0) == -1
    assert merge_absorb(H=65536) == -1
    assert merge_absorb(od=2) == -1
    assert merge_absorb(vd=7) == -1
    assert merge_absorb(base=2) == -1
    assert merge_absorb(lp=None) == -1
    assert merge_absorb(w=P(520)) == -1             # not 16-byte aligned
    # the exchange of the partials over W ranks
    assert lib.dcp_a2a_chunk_bytes(1, 64, 96, 8, 1) > 0
    assert lib.dcp_a2a_chunk_bytes(1, 64, 96, 7, 1) == 0    # heads do not split evenly
    assert lib.dcp_a2a_chunk_bytes(0, 64, 96, 8, 1) == 0
    assert lib.dcp_a2a_chunk_bytes(1, 64, 96, 8, 5) == 0

    def pack(nh=1, T=4, H=8, W=2, o=P(256), od=0, lp=P(256), send=P(1024), wd=1):
        return lib.dcp_pack_partials(nh, T, H, W, o, od, lp, send, wd, None)
    assert pack(T=0) == 0
    assert pack(W=3) == -1
    assert pack(od=4) == -1
    assert pack(send=None) == -1
    assert pack(o=P(264)) == -1

    def merge_packed(W=2, nh=1, rows=16, recv=P(1024), wd=1, base=0, o=P(256), od=1):
        return lib.dcp_lse_merge_packed(W, nh, rows, recv, wd, base, o, od, None, None)
    assert merge_packed(rows=0) == 0
    assert merge_packed(W=0) == -1
    assert merge_packed(nh=0) == -1
    assert merge_packed(base=3) == -1
    assert merge_packed(recv=None) == -1
    assert merge_packed(o=P(260)) == -1

    def rescale(N=8, sb=0, nh=4, T=4, H=8, W=2, la=P(256), o=P(512), od=0, base=0, os=P(1024)):
        return lib.dcp_lse_rescale(N, sb, nh, T, H, W, la, o, od, base, os, None, None)
    assert rescale(T=0) == 0
    assert rescale(sb=6) == -1                      # shards [6, 10) past the 8 shards
    assert rescale(W=3) == -1
    assert rescale(base=5) == -1
    assert rescale(la=None) == -1
    assert rescale(os=P(1028)) == -1


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    import context_sharded_mla_gb300 as dcp
    monkeypatch.setattr(dcp, "_lib", None)
    monkeypatch.setattr(dcp._build, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        dcp.load_library()
