"""GPU parity of dcp_absorb_q / dcp_absorb_o (the absorption products) against the oracle.

Bars: |err| <= 1e-2 + 1e-2 |ref| against the fp64 oracle on the same bf16
inputs, and the 64 rope dims copied bit for bit.  Cases: the K3 shapes (64
tokens x 96 heads) with q_nope / q_pe as slices of one [.., 192] projection,
ragged token tails (1, 129 and 300 tokens: one, two and three 128-token tiles),
q_len = 4 leading dims, f32 and bf16 o / v, and the whole absorbed layer
(absorb_q -> append -> partial -> merge -> absorb_o) against the oracle's
absorbed attention.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import absorb as oabsorb
from harness import GpuState, assert_close_o, bits, to_f64

pytestmark = pytest.mark.gpu


def lib():
    import context_sharded_mla_gb300 as dcp
    return dcp


def run_q(q_nope, q_pe, w_kc):
    dcp = lib()
    q = torch.full(q_nope.shape[:-1] + (576,), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.dcp_absorb_q(q_nope, q_pe, w_kc, q, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return q


def check_q(q, q_nope, q_pe, w_kc, what):
    ref = oabsorb.absorb_q(to_f64(q_nope), to_f64(w_kc))
    assert_close_o(to_f64(q[..., :512]), ref, what)
    assert np.array_equal(bits(q[..., 512:]), bits(q_pe.contiguous())), f"{what}: rope dims not copied exactly"


def test_absorb_q_k3_shape_from_projection():
    cfg = workloads.config("k3")
    qp = workloads.gen_q_proj(cfg).to("cuda")            # [64, 1, 96, 192]
    w_kc, _ = workloads.gen_absorb_weights(cfg)
    w_kc = w_kc.to("cuda")
    q_nope, q_pe = qp[..., :128], qp[..., 128:]
    q = run_q(q_nope, q_pe, w_kc)
    check_q(q, q_nope, q_pe, w_kc, "absorb_q k3")


@pytest.mark.parametrize("B,q_len,H", [(1, 1, 3), (129, 1, 2), (75, 4, 5), (300, 1, 1)])
def test_absorb_q_ragged_token_tiles(B, q_len, H):
    cfg = workloads.config("tiny", B=B, q_len=q_len, H=H, seed=B + H)
    qp = workloads.gen_q_proj(cfg).to("cuda")
    w_kc, _ = workloads.gen_absorb_weights(cfg)
    q_nope = qp[..., :128].contiguous()                  # stride 128 rows
    q_pe = qp[..., 128:].contiguous()                    # stride 64 rows
    q = run_q(q_nope, q_pe, w_kc.to("cuda"))
    check_q(q, q_nope, q_pe, w_kc.to("cuda"), f"absorb_q B={B} q_len={q_len} H={H}")


def run_o(o, w_vc, v_dtype):
    dcp = lib()
    v = torch.full(o.shape[:-1] + (128,), float("nan"), dtype=v_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.dcp_absorb_o(o, w_vc, v, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return v


def check_o(v, o, w_vc, what):
    """Parity bar against the oracle on the operand the kernel multiplies (an f32
    o rounded to nearest bf16, as the ABI states); and against the exact o within
    the rounding bound of that operand, 2^-8 sum_k |o_k w_k| (bf16 keeps 8
    significant bits), plus the bf16 output rounding when v is bf16."""
    w = to_f64(w_vc)
    o_op = to_f64(o.to(torch.bfloat16))
    got = to_f64(v)
    assert_close_o(got, oabsorb.absorb_o(o_op, w), what)
    exact = oabsorb.absorb_o(to_f64(o), w)
    mag = oabsorb.absorb_o(np.abs(to_f64(o)), np.abs(w))
    bound = 2.0 ** -8 * mag * 1.001 + 1e-6
    if v.dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(exact) + bound)
    err = np.abs(got - exact)
    assert np.all(err <= bound), f"{what}: max err / bound {np.max(err / bound):.3f} against the exact o"


@pytest.mark.parametrize("o_dtype,v_dtype", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                             (torch.float32, torch.bfloat16), (torch.bfloat16, torch.float32)])
def test_absorb_o_k3_shape(o_dtype, v_dtype):
    cfg = workloads.config("k3")
    _, w_vc = workloads.gen_absorb_weights(cfg)
    g = torch.Generator().manual_seed(77)
    o = torch.randn(cfg.B, cfg.q_len, cfg.H, 512, generator=g).to(o_dtype)
    v = run_o(o.to("cuda"), w_vc.to("cuda"), v_dtype)
    check_o(v, o, w_vc, f"absorb_o k3 {o_dtype}->{v_dtype}")


@pytest.mark.parametrize("T,H", [(1, 1), (129, 3), (300, 2), (200, 7)])
def test_absorb_o_ragged_token_tiles(T, H):
    g = torch.Generator().manual_seed(T * 31 + H)
    o = torch.randn(T, H, 512, generator=g) * 3.0
    w_vc = (torch.randn(H, 512, 128, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    v = run_o(o.to("cuda"), w_vc.to("cuda"), torch.float32)
    check_o(v, o, w_vc, f"absorb_o T={T} H={H}")


def test_absorbed_layer_end_to_end():
    """absorb_q -> owner-filtered append -> partials -> merge -> absorb_o on the
    GPU against the oracle's absorbed query, sharded attention and o @ w_vc, all
    from the same seeded bf16 inputs."""
    cfg = workloads.config("tiny", B=2, H=16, S=1000, seed=12)
    st = GpuState(cfg)
    qp = workloads.gen_q_proj(cfg).to("cuda")
    w_kc, w_vc = workloads.gen_absorb_weights(cfg)
    w_kc, w_vc = w_kc.to("cuda"), w_vc.to("cuda")
    q = run_q(qp[..., :128], qp[..., 128:], w_kc)
    o, _lse = st.dec.decode(q, st.bt, st.seq_lens)
    torch.cuda.synchronize()
    v = run_o(o.view(cfg.B, cfg.q_len, cfg.H, 512), w_vc, torch.float32)
    q_ref = oabsorb.absorbed_query(to_f64(qp[..., :128]), to_f64(qp[..., 128:]), to_f64(w_kc))
    from oracle import attention
    for b in range(cfg.B):
        o_ref, _l, _op, _lp = attention.sharded_attention(q_ref[b], to_f64(st.kv[b]), int(st.S[b]), cfg.N, cfg.I,
                                                          workloads.SCALE, cfg.base)
        v_ref = oabsorb.absorb_o(o_ref, to_f64(w_vc))
        assert_close_o(to_f64(v[b]), v_ref, f"absorbed layer b={b}")


def test_absorb_fails_loudly_on_bad_views():
    dcp = lib()
    w_kc = torch.zeros(4, 128, 512, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(8, 4, 576, dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros(8, 4, 192, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        dcp.dcp_absorb_q(qp[..., :128].float(), qp[..., 128:], w_kc, q)
    with pytest.raises(ValueError):
        dcp.dcp_absorb_q(qp.transpose(0, 1)[..., :128], qp[..., 128:], w_kc, q)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_absorb_q(qp[..., 1:129], qp[..., 128:], w_kc, q)      # base not 16-byte aligned
