"""GPU parity of dcp_lse_merge_absorb_o (the merge and the output-side product in
one kernel) against the oracle's merge followed by o @ w_vc.

The kernel rounds the merged o to nearest bf16 before the product (the tensor
core multiplies bf16 by bf16), so v is compared with the oracle on the exact
merged o within the rounding bound of that operand, 2^-8 sum_k |o_k w_kn|, plus
the bf16 output rounding when v is bf16; lse within 1e-5 of the oracle's merge.
Cases: the K3 shapes (8 parts, 64 tokens, 96 heads, base 2), 16 parts, one
part, 64 parts (the most the call takes), token tails of 1, 20, 33 and 300
tokens (the kernel's items are 16 tokens of one head), bf16 partials, empty parts (lse = -inf) and a row whose parts are all empty,
and the absorbed decode layer end to end.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import absorb as oabsorb, attention
from harness import GpuState, assert_close_o, to_f64

pytestmark = pytest.mark.gpu


def make_parts(n, T, H, part_dtype, seed, empty_frac=0.0):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(n, T, H, 512, generator=g).to(part_dtype)
    lse = torch.randn(n, T, H, generator=g) * 3.0
    if empty_frac:
        drop = torch.rand(n, T, H, generator=g) < empty_frac
        lse[drop] = float("-inf")
        o[drop] = 0
    return o, lse


def run(o, lse, w_vc, base, v_dtype):
    import context_sharded_mla_gb300 as dcp
    T, H = o.shape[1], o.shape[2]
    v = torch.full((T, H, 128), float("nan"), dtype=v_dtype, device="cuda")
    lse_out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.dcp_lse_merge_absorb_o(o.cuda(), lse.cuda(), 1 if base == 2 else 0, w_vc.cuda(), v, lse_out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return v, lse_out


def check(v, lse_out, o, lse, w_vc, base, what):
    o_m, l_m = attention.merge(to_f64(o), to_f64(lse), base)        # the exact merged o and lse
    w = to_f64(w_vc)
    exact = oabsorb.absorb_o(o_m, w)
    bound = 2.0 ** -8 * oabsorb.absorb_o(np.abs(o_m), np.abs(w)) * 1.001 + 1e-5
    got = to_f64(v)
    if v.dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(exact) + bound)
    assert np.all(np.isfinite(got)), f"{what}: non-finite v"
    err = np.abs(got - exact)
    assert np.all(err <= bound), f"{what}: max err / bound {np.max(err / bound):.3f}"
    lg = to_f64(lse_out)
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_m)), f"{what}: -inf pattern of lse differs"
    fin = ~np.isneginf(l_m)
    if fin.any():
        assert np.max(np.abs(lg[fin] - l_m[fin])) <= 1e-5, f"{what}: lse"


@pytest.mark.parametrize("part_dtype,v_dtype,base", [(torch.float32, torch.bfloat16, 2),
                                                     (torch.float32, torch.float32, 0),
                                                     (torch.bfloat16, torch.bfloat16, 2),
                                                     (torch.bfloat16, torch.float32, 0)])
def test_merge_absorb_k3_shapes(part_dtype, v_dtype, base):
    cfg = workloads.config("k3")
    _, w_vc = workloads.gen_absorb_weights(cfg)
    o, lse = make_parts(cfg.N, cfg.B, cfg.H, part_dtype, seed=3, empty_frac=0.1)
    v, lse_out = run(o, lse, w_vc, base, v_dtype)
    check(v, lse_out, o, lse, w_vc, base, f"k3 {part_dtype}->{v_dtype} base {base}")


@pytest.mark.parametrize("n,T,H", [(16, 33, 5), (1, 300, 2), (8, 1, 3), (3, 64, 1), (64, 20, 2)])
def test_merge_absorb_token_tails_and_part_counts(n, T, H):
    g = torch.Generator().manual_seed(n * 1000 + T)
    w_vc = (torch.randn(H, 512, 128, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    o, lse = make_parts(n, T, H, torch.float32, seed=n + T, empty_frac=0.2 if n > 1 else 0.0)
    v, lse_out = run(o, lse, w_vc, 0, torch.float32)
    check(v, lse_out, o, lse, w_vc, 0, f"n={n} T={T} H={H}")


def test_merge_absorb_all_empty_row():
    g = torch.Generator().manual_seed(9)
    w_vc = (torch.randn(4, 512, 128, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    o, lse = make_parts(8, 40, 4, torch.float32, seed=9)
    lse[:, 7, 2] = float("-inf")                            # token 7, head 2: no part has a key
    o[:, 7, 2] = 0
    v, lse_out = run(o, lse, w_vc, 2, torch.float32)
    assert torch.all(v[7, 2] == 0) and torch.isneginf(lse_out[7, 2])
    check(v, lse_out, o, lse, w_vc, 2, "all-empty row")


def test_absorbed_layer_with_the_fused_merge():
    """absorb_q -> append -> partials -> dcp_lse_merge_absorb_o, against the
    oracle's absorbed query, sharded attention and o @ w_vc."""
    import context_sharded_mla_gb300 as dcp
    cfg = workloads.config("k3", B=3, S=3000, seed=13)
    st = GpuState(cfg)
    qp = workloads.gen_q_proj(cfg).to("cuda")
    w_kc, w_vc = workloads.gen_absorb_weights(cfg)
    w_kc, w_vc = w_kc.to("cuda"), w_vc.to("cuda")
    q = torch.empty(cfg.B, cfg.q_len, cfg.H, 576, dtype=torch.bfloat16, device="cuda")
    dcp.dcp_absorb_q(qp[..., :128], qp[..., 128:], w_kc, q)
    st.dec.partial(q, st.bt, st.seq_lens)
    v = torch.empty(cfg.B, cfg.q_len, cfg.H, 128, dtype=torch.float32, device="cuda")
    lse = torch.empty(cfg.B, cfg.q_len, cfg.H, dtype=torch.float32, device="cuda")
    dcp.dcp_lse_merge_absorb_o(st.dec.o_part, st.dec.lse_part, 1, w_vc, v, lse)
    torch.cuda.synchronize()
    assert st.dec.status_bits() == 0
    q_ref = oabsorb.absorbed_query(to_f64(qp[..., :128]), to_f64(qp[..., 128:]), to_f64(w_kc))
    # the decode call takes a bf16 query: round the oracle's absorbed query the same way
    q_ref = torch.from_numpy(q_ref).to(torch.bfloat16).double().numpy()
    for b in range(cfg.B):
        o_ref, l_ref, _op, _lp = attention.sharded_attention(q_ref[b], to_f64(st.kv[b]), int(st.S[b]), cfg.N,
                                                             cfg.I, workloads.SCALE, cfg.base)
        assert_close_o(to_f64(v[b]), oabsorb.absorb_o(o_ref, to_f64(w_vc)), f"fused layer v b={b}")
        assert np.max(np.abs(to_f64(lse[b]) - l_ref)) <= 1e-3
