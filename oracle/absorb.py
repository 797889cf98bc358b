"""Oracle: the two absorption products around the decode path (fp64, CPU).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "MLA 的 Decode Context Parallelism", section 2 "吸收形式：decode 实际
执行的东西":
  identity (1), the K up-projection moved to the query side:
      q^C . (W^UK_h c) = (q^C . W^UK_h) . c,  q_hat_h = q^C . W^UK_h in R^512;
  identity (2), the V up-projection applied after attention:
      sum_t a_t (W^UV_h c_t) = W^UV_h (sum_t a_t c_t),  u_hat_h in R^512;
and "Decode Context Parallelism" (zdszero), section "decode 路径：以 Kimi K3
的 MLA 为例" (the per-card shapes of one layer): w_kc [H, 128, 512] is the K
part of kv_b_proj, so w_kc[h] = W^UK_h (128 x 512); w_vc [H, 512, 128] is the
V part, w_vc[h] = (W^UV_h)^T.  The query side is bmm(q_nope, w_kc) ->
[B, H, 512] and the output side bmm(O, w_vc) -> [B, H, 128].  The absorbed
query of head h is [q_hat_h || q_pe_h] (576 dims); the 64-d rope part passes
through unchanged (K3 builds its MLA without rotary embedding).

Both functions are the plain per-head matrix products of those identities.
"""

from __future__ import annotations

import numpy as np


def absorb_q(q_nope, w_kc):
    """q_hat [..., H, 512] = per head q_nope [..., H, 128] @ w_kc[h] [128, 512].

    Leading dims are the query tokens (B, or B x q_len)."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    w_kc = np.asarray(w_kc, dtype=np.float64)
    return np.einsum("...hk,hkn->...hn", q_nope, w_kc)


def absorb_o(o, w_vc):
    """v [..., H, 128] = per head o [..., H, 512] @ w_vc[h] [512, 128]."""
    o = np.asarray(o, dtype=np.float64)
    w_vc = np.asarray(w_vc, dtype=np.float64)
    return np.einsum("...hk,hkn->...hn", o, w_vc)


def absorbed_query(q_nope, q_pe, w_kc):
    """The 576-d query of each head: [absorb_q(q_nope) || q_pe]."""
    return np.concatenate([absorb_q(q_nope, w_kc), np.asarray(q_pe, dtype=np.float64)], axis=-1)
