"""Test harness: seeded workloads on the GPU (through the C ABI) and oracle references.

Inputs come from ``workloads`` only.  The GPU side places them with the
library's own slot map + append; the oracle side reads the same input rows
(never anything the CUDA path produced) and computes its reference in fp64.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import workloads
from oracle import attention, layout as olayout


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class GpuState:
    """A workload appended into a ShardedMlaDecoder (inputs kept for the oracle)."""

    def __init__(self, cfg, gen_device="cpu", needle=False, part_dtype=torch.float32, keep_kv=True,
                 out_dtype=None):
        from context_sharded_mla_gb300 import Layout
        from context_sharded_mla_gb300.step import ShardedMlaDecoder

        self.cfg = cfg
        self.gen_device = gen_device
        dev = torch.device("cuda")
        self.S = workloads.lengths(cfg)
        self.bt_cpu, self.pool_pages = workloads.block_table(cfg, self.S)
        self.max_pages = self.bt_cpu.shape[1]
        self.layout = Layout(cfg.N, cfg.I, cfg.P)
        self.q = workloads.gen_q(cfg, gen_device).to(dev)
        self.bt = self.bt_cpu.to(dev)
        self.seq_lens = self.S.to(dev)
        od = out_dtype or (torch.float32 if cfg.out_dtype == "f32" else torch.bfloat16)
        self.dec = ShardedMlaDecoder(self.layout, cfg.B, cfg.q_len, cfg.H, self.pool_pages, self.max_pages,
                                     workloads.SCALE, 1 if cfg.base == 2 else 0, od, part_dtype)
        self.needle_pos = workloads.needle_positions(cfg, self.S) if needle else None
        self.kv = {}
        for b in range(cfg.B):
            kv_b = self.kv_request(b)
            if keep_kv:
                self.kv[b] = kv_b.cpu()
            S_b = int(self.S[b])
            pos = torch.arange(S_b, dtype=torch.int64, device=dev)
            req = torch.full((S_b,), b, dtype=torch.int32, device=dev)
            self.dec.append(kv_b.to(dev), pos, req, self.bt)
        torch.cuda.synchronize()

    def kv_request(self, b):
        """Request b's latent rows in position order (regenerated from the seed)."""
        kv_b = workloads.gen_kv(self.cfg, b, int(self.S[b]), self.gen_device)
        if self.needle_pos is not None:
            workloads.plant_needle(self.q.to(kv_b.device), kv_b, b, int(self.needle_pos[b]), head=b % self.cfg.H)
        return kv_b

    def decode(self):
        o, lse = self.dec.decode(self.q, self.bt, self.seq_lens)
        torch.cuda.synchronize()
        return o, lse

    def oracle_request(self, b, heads=None):
        """fp64 oracle (merged o, lse, per-shard o_parts, lse_parts) for request b."""
        cfg = self.cfg
        kv_b = self.kv[b] if b in self.kv else self.kv_request(b).cpu()
        q_b = to_f64(self.q[b])
        if heads is not None:
            q_b = q_b[:, heads]
        return attention.sharded_attention(q_b, to_f64(kv_b), int(self.S[b]), cfg.N, cfg.I,
                                           workloads.SCALE, cfg.base)


def assert_close_o(got, ref, what, atol=1e-2, rtol=1e-2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside |err| <= {atol} + {rtol}|ref|; "
                           f"max err {err.max():.3e}")


def assert_close_lse(got, ref, what, atol=1e-3):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= atol, f"{what}: lse max err {err.max():.3e} > {atol}"


def rel_row_err(got, ref):
    """max over rows of ||got - ref|| / ||ref|| (reported next to the elementwise bound)."""
    got = np.asarray(got, np.float64).reshape(-1, 512)
    ref = np.asarray(ref, np.float64).reshape(-1, 512)
    n = np.linalg.norm(ref, axis=1)
    keep = n > 0
    if not keep.any():
        return 0.0
    return float(np.max(np.linalg.norm(got - ref, axis=1)[keep] / n[keep]))


__all__ = ["GpuState", "assert_close_o", "assert_close_lse", "rel_row_err", "to_f64", "bits", "olayout", "math"]
