"""Seeded synthetic inputs for sharded MLA decode (shared by the oracle side and the CUDA side).

This module only draws inputs: shapes, lengths, block tables, query and latent
rows.  It holds none of the method's arithmetic (no ownership, slot, softmax or
merge computation); the oracle and the CUDA library each do that on their own.

Workloads (all bf16 latent rows of 576 = 512 c_K + 64 k_R dims drawn from N(0,1),
queries from N(0,1), softmax scale 1/sqrt(192), shuffled block tables):

  tiny    B=1,   H=16,  q_len=1, S=1024,                 N=4,  I=1,  P=16, base e, fp32 out
  dsv3    B=32,  H=128, q_len=1, S=32768,                N=8,  I=1,  P=64, base e
  k3      B=64,  H=96,  q_len=1, S=131072, +1-token append, N=8, I=1, P=64, base 2
  ragged  B=128, H=128, q_len=4 (causal), S_b log-uniform in [1024, 262144], N=16, I=16, P=64, base e
  long    B=4,   H=96,  q_len=1, S=1048576, +8192-token chunk append at a=S-8192, N=8, I=1, P=64, base e
  extend  B=4,   H=96,  q_len=64 (causal), S=131072, +64-token chunk append, N=8, I=1, P=64, base e
          (a chunked extend in the all-gather-Q form: the chunk's 64 tokens are the query rows)

Capacity: the pool is sized with the widened-page rule of the SGLang page
"Decode context parallelism" ("Virtual KV layout"): one virtual page covers
N*P request positions and maps to one physical page of P rows on each shard,
so a request of S tokens is given ceil(S / (N*P)) pages, shared by all shards.
The block table is a seeded random permutation of the pool's pages.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

SCALE = 1.0 / math.sqrt(192.0)
DK = 576
DV = 512

_BASE = {
    "tiny": dict(B=1, H=16, q_len=1, S=1024, N=4, I=1, P=16, base=0, out_dtype="f32",
                 seed=1, append=0, chunk=0, ragged=False),
    "dsv3": dict(B=32, H=128, q_len=1, S=32768, N=8, I=1, P=64, base=0, out_dtype="bf16",
                 seed=2, append=0, chunk=0, ragged=False),
    "k3": dict(B=64, H=96, q_len=1, S=131072, N=8, I=1, P=64, base=2, out_dtype="bf16",
               seed=3, append=1, chunk=0, ragged=False),
    "ragged": dict(B=128, H=128, q_len=4, S=262144, S_min=1024, N=16, I=16, P=64, base=0,
                   out_dtype="bf16", seed=4, append=0, chunk=0, ragged=True),
    "long": dict(B=4, H=96, q_len=1, S=1048576, N=8, I=1, P=64, base=0, out_dtype="bf16",
                 seed=5, append=0, chunk=8192, ragged=False),
    "extend": dict(B=4, H=96, q_len=64, S=131072, N=8, I=1, P=64, base=0, out_dtype="bf16",
                   seed=6, append=0, chunk=64, ragged=False),
}

DESCRIPTIONS = {
    "tiny": "tiny: B=1 H=16 q_len=1 S=1024 N=4 RR page16 base-e fp32 out",
    "dsv3": "DeepSeek-V3-shaped: B=32 H=128 S=32768 N=8 RR page64 base-e",
    "k3": "K3-shaped: B=64 H=96 S=131072 N=8 RR page64 base-2 +1-token owner-filtered append",
    "ragged": "ragged verify: B=128 H=128 q_len=4 causal S~logU[1k,256k] N=16 I=16 page64 base-e",
    "long": "long context: B=4 H=96 S=1048576 N=8 RR page64 base-e +8192-token chunk append",
    "extend": "chunked extend (all-gather-Q): B=4 H=96 q_len=64 causal S=131072 N=8 RR page64 base-e "
              "+64-token chunk append",
}


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    H: int
    q_len: int
    S: int              # length of every request (max length when ragged)
    N: int              # context shards
    I: int              # interleave size (1 = token round-robin)
    P: int              # physical page size (rows)
    base: int           # 0 = natural-log LSE, 2 = log2 LSE
    out_dtype: str      # "f32" or "bf16" for the merged output
    seed: int
    append: int = 0     # tokens appended per request each step (decode)
    chunk: int = 0      # tokens appended per request each step (chunked append)
    ragged: bool = False
    S_min: int = 0      # lower end of the log-uniform length draw when ragged
    lengths_override: tuple = field(default=None)
    needle: bool = False

    @property
    def rows(self):
        return self.B * self.q_len * self.H


def config(name: str, **overrides) -> Config:
    """A named workload, optionally reshaped (smaller B/S/H for parity tests)."""
    base_name = name
    d = dict(_BASE[base_name])
    cfg = Config(name=name, **d)
    if overrides:
        cfg = replace(cfg, **overrides)
    return cfg


def lengths(cfg: Config) -> torch.Tensor:
    """Per-request token counts S_b (the tokens appended this step included)."""
    if cfg.lengths_override is not None:
        return torch.tensor(cfg.lengths_override, dtype=torch.int64)
    if not cfg.ragged:
        return torch.full((cfg.B,), cfg.S, dtype=torch.int64)
    g = torch.Generator().manual_seed(cfg.seed * 7919 + 11)
    u = torch.rand(cfg.B, generator=g, dtype=torch.float64)
    lo, hi = math.log(cfg.S_min), math.log(cfg.S)
    L = torch.floor(torch.exp(lo + u * (hi - lo))).to(torch.int64)
    return torch.clamp(L, min=max(cfg.q_len, 1), max=cfg.S)


def pages_per_request(cfg: Config, S_b: torch.Tensor) -> torch.Tensor:
    """Physical pages given to each request (widened-page capacity rule)."""
    per_page = cfg.N * cfg.P
    return torch.clamp((S_b + per_page - 1) // per_page, min=1)


def block_table(cfg: Config, S_b: torch.Tensor, spare_pages: int = 0):
    """(bt int32 [B, max_pages] padded with -1, pool_pages): a shuffled page assignment."""
    npages = pages_per_request(cfg, S_b)
    pool_pages = int(npages.sum()) + spare_pages
    max_pages = int(npages.max())
    g = torch.Generator().manual_seed(cfg.seed * 104729 + 3)
    perm = torch.randperm(pool_pages, generator=g).to(torch.int32)
    bt = torch.full((cfg.B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(cfg.B):
        n = int(npages[b])
        bt[b, :n] = perm[off: off + n]
        off += n
    return bt, pool_pages


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def gen_q(cfg: Config, device="cpu") -> torch.Tensor:
    """Absorbed queries [B, q_len, H, 576] bf16 from N(0,1)."""
    g = _gen(device, cfg.seed * 1000003 + 17)
    q = torch.randn(cfg.B, cfg.q_len, cfg.H, DK, generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16)


def gen_q_proj(cfg: Config, device="cpu") -> torch.Tensor:
    """Per-head query projection [B, q_len, H, 192] bf16 from N(0,1): dims [0, 128)
    are q_nope, dims [128, 192) are q_pe (the input of the query-side absorption)."""
    g = _gen(device, cfg.seed * 1000003 + 29)
    q = torch.randn(cfg.B, cfg.q_len, cfg.H, 192, generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16)


def gen_absorb_weights(cfg: Config, device="cpu"):
    """Synthetic (w_kc [H, 128, 512], w_vc [H, 512, 128]) bf16 with entries drawn
    from N(0, 1/fan_in) (fan_in 128 and 512), so q_nope @ w_kc has unit-variance
    dims like the other query recipes and o @ w_vc stays on the scale of o."""
    g = _gen(device, cfg.seed * 1000003 + 31)
    w_kc = torch.randn(cfg.H, 128, DV, generator=g, device=device, dtype=torch.float32) / math.sqrt(128.0)
    w_vc = torch.randn(cfg.H, DV, 128, generator=g, device=device, dtype=torch.float32) / math.sqrt(512.0)
    return w_kc.to(torch.bfloat16), w_vc.to(torch.bfloat16)


def gen_kv(cfg: Config, b: int, S_b: int, device="cpu") -> torch.Tensor:
    """Latent rows [S_b, 576] bf16 of request b in position order, from N(0,1)."""
    g = _gen(device, cfg.seed * 1000003 + 1009 * (b + 1))
    kv = torch.randn(S_b, DK, generator=g, device=device, dtype=torch.float32)
    return kv.to(torch.bfloat16)


def needle_positions(cfg: Config, S_b: torch.Tensor) -> torch.Tensor:
    """One seeded position per request for a planted 'needle' row (visible to every query token)."""
    g = torch.Generator().manual_seed(cfg.seed * 31337 + 5)
    u = torch.rand(cfg.B, generator=g, dtype=torch.float64)
    p = (u * S_b.to(torch.float64)).to(torch.int64)
    return torch.clamp(torch.minimum(p, S_b - cfg.q_len), min=0)


def plant_needle(q: torch.Tensor, kv_b: torch.Tensor, b: int, p: int, head: int = 0):
    """Copy query row (t=0, head) of request b into latent row p (in place).

    That row then scores about |q|^2 / sqrt(192) ~ 40 for that head, so one
    token (and so one shard) carries almost all of the softmax weight and the
    output is O(1) instead of O(1/sqrt(S)).
    """
    kv_b[p] = q[b, 0, head]
    return kv_b


def edge_lengths(cfg: Config):
    """Lengths 1 .. N*I + 1 (cycled over B): short requests leave some shards empty."""
    top = cfg.N * cfg.I + 1
    return tuple(max(cfg.q_len, 1 + (b % top)) for b in range(cfg.B))
