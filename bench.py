"""Benchmark: sharded absorbed-MLA decode + LSE merge on GB300 (one JSON line).

A step is one pass of the whole hot path over one batch of the workload:
slot map + owner-filtered append of this step's new tokens, the per-shard
partials of every shard, and the LSE merge.  The default workload is the
K3-shaped configuration (B=64, H=96, S=131072, N=8 token round-robin shards,
page 64, base-2 LSE, one appended token per request per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload k3|dsv3|ragged|long|tiny|extend]
                  [--op decode|relayout|absorb] [--exchange a2a|ag_rs] [--group]
                  [--impl ours|reference] [--batch B] [--no-cpu-baseline] [--no-e2e]

`value` is KV-read GB/s (sum over requests of S_b * 1152 bytes per step,
divided by the device time per step).  With --gpus N > 1 (under torchrun) the
same step runs as Decode Context Parallelism over the N GPUs: each rank holds
N_shards / N of the shards, computes their partials for all heads, and the
partials are exchanged over NCCL (--exchange a2a: packed all-to-all by head
slice and a local merge; ag_rs: AllGather of the lse + ReduceScatter) so that
each rank ends with the merged output of H / N heads; total work is fixed
(strong scaling) and `value` is the whole job's KV GB/s over the slowest rank's
step time.  --impl reference times the fp64 CPU oracle on a bounded sample of
the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "sharded MLA decode+merge: µs/step, KV-read GB/s, % of binding roofline"
KV_ROW_BYTES = 576 * 2
FLOP_PER_TOKEN_ROW = 2 * (576 + 512)


# ----------------------------------------------------------------------------- helpers

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device_sync=True):
    if device_sync and torch.cuda.is_available():
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_accounting(cfg, S_b):
    """Algorithmic bytes and FLOPs of one step (what the method must move / compute)."""
    S = [int(s) for s in S_b]
    R = cfg.q_len * cfg.H
    kv_bytes = sum(S) * KV_ROW_BYTES
    q_bytes = cfg.B * R * 576 * 2
    parts = cfg.N * cfg.B * R
    part_bytes = parts * (512 * 2 + 4) * 2          # bf16 o_r + fp32 lse, written once and read once
    out_bytes = cfg.B * R * (512 * (4 if cfg.out_dtype == "f32" else 2) + 4)
    new_tokens = cfg.B * max(cfg.append, cfg.chunk)
    append_bytes = new_tokens * KV_ROW_BYTES * 2
    # FLOPs: every visible (token, row) pair, causal rows see S_b - q_len + t + 1 tokens
    flops = 0
    for s in S:
        for t in range(cfg.q_len):
            flops += (s - cfg.q_len + t + 1) * cfg.H * FLOP_PER_TOKEN_ROW
    # the partial call's own algorithmic bytes: KV and Q read once, each partial
    # summary written once at the pages' minimum (bf16 o_r + fp32 lse_r)
    return {"kv_bytes": kv_bytes, "bytes_alg": kv_bytes + q_bytes + part_bytes + out_bytes + append_bytes,
            "flops_alg": flops, "partial_bytes_alg": kv_bytes + q_bytes + parts * (512 * 2 + 4)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join(os.environ.get("DCP_CLOCK_LOG_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self):
        """Host time at the edge of the timed region (the sampler keeps only samples between marks)."""
        self.marks = getattr(self, "marks", []) + [time.time()]

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        return self.summarize()

    def summarize(self):
        """Median / minimum SM clock and the throttle reasons seen between the marks."""
        import datetime
        lo, hi = (self.marks[0], self.marks[-1]) if len(getattr(self, "marks", [])) >= 2 else (None, None)
        sm, mx, reasons, all_sm = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, cmax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                all_sm.append(clk)
                # samples inside the timed region (100 ms sampling: allow one period of slack)
                if lo is not None and not (lo - 0.1 <= ts <= hi + 0.1):
                    continue
                sm.append(clk)
                mx.append(cmax)
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "sm_mhz_min": min(sm), "reasons": sorted(reasons), "window": "timed region only"}


# ----------------------------------------------------------------------------- our arm

def build_state(cfg, device, rank=0, world=1, strategy=None, part_dtype=torch.float32):
    """The workload's cache appended into this rank's decoder: all N shards on one
    GPU (world == 1), or, with a DCP group, this rank's N / world shards."""
    import context_sharded_mla_gb300 as dcp
    from context_sharded_mla_gb300.step import ShardedMlaDecoder
    dcp.load_library()
    S = workloads.lengths(cfg)
    bt, pool_pages = workloads.block_table(cfg, S)
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    new = max(cfg.append, cfg.chunk)
    out_dtype = torch.float32 if cfg.out_dtype == "f32" else torch.bfloat16
    base = dcp.DCP_LSE_BASE_2 if cfg.base == 2 else dcp.DCP_LSE_BASE_E
    if strategy is None:
        dec = ShardedMlaDecoder(lay, cfg.B, cfg.q_len, cfg.H, pool_pages, bt.shape[1], workloads.SCALE, base,
                                out_dtype, part_dtype, device=device)
    else:
        from context_sharded_mla_gb300.group import DcpGroupDecoder
        dec = DcpGroupDecoder(lay, cfg.B, cfg.q_len, cfg.H, pool_pages, bt.shape[1], workloads.SCALE, rank, world,
                              base, strategy, torch.bfloat16, out_dtype, part_dtype, device=device)
    btd = bt.to(device)
    # cache: every request holds S_b - new tokens before the step; the step appends the rest
    new_rows, new_pos, new_req = [], [], []
    for b in range(cfg.B):
        S_b = int(S[b])
        kv_b = workloads.gen_kv(cfg, b, S_b, device)
        pre = S_b - new
        dec.append(kv_b[:pre].contiguous(), torch.arange(pre, device=device),
                   torch.full((pre,), b, dtype=torch.int32, device=device), btd)
        if new:
            new_rows.append(kv_b[pre:].clone())
            new_pos.append(torch.arange(pre, S_b, device=device))
            new_req.append(torch.full((new,), b, dtype=torch.int32, device=device))
        del kv_b
    torch.cuda.synchronize()
    st = {"dec": dec, "bt": btd, "S": S, "seq_lens": S.to(device), "q": workloads.gen_q(cfg, device),
          "pool_pages": pool_pages}
    if new:
        st["kv_new"] = torch.cat(new_rows).contiguous()
        st["pos"] = torch.cat(new_pos).contiguous()
        st["req"] = torch.cat(new_req).contiguous()
    else:
        st["kv_new"] = st["pos"] = st["req"] = None
    return st


def held_kv_rows(cfg, S, shard_begin, shard_end):
    """KV rows of shards [shard_begin, shard_end) over all requests (the library's count)."""
    import context_sharded_mla_gb300 as dcp
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    return sum(dcp.dcp_count(lay, r, int(s)) for s in S for r in range(shard_begin, shard_end))


def run_ours(args, cfg, rank, world, dist, device):
    import context_sharded_mla_gb300 as dcp
    group = world > 1 or args.group
    if group:
        # Decode Context Parallelism over the ranks: N / world shards per GPU, heads
        # split H / world per GPU after the exchange; total work fixed (strong scaling)
        if cfg.N % world or cfg.H % world:
            raise SystemExit(f"{cfg.name}: {cfg.N} shards and {cfg.H} heads must split evenly over {world} GPUs")
    part_dtype = torch.bfloat16 if args.partials == "bf16" else torch.float32
    st = build_state(cfg, device, rank, world, args.exchange if group else None, part_dtype)
    dec = st["dec"]
    acct = workload_accounting(cfg, st["S"])
    if group:
        sb, se = dec.local.shard_begin, dec.local.shard_end
        n_held = se - sb
        R = cfg.q_len * cfg.H
        # this rank's share of the partial call: its shards' KV, the replicated query, its partial summaries
        acct["partial_bytes_alg"] = (held_kv_rows(cfg, st["S"], sb, se) * KV_ROW_BYTES + cfg.B * R * 576 * 2
                                     + n_held * cfg.B * R * (512 * 2 + 4))
        acct["flops_alg_rank"] = acct["flops_alg"] * n_held / cfg.N
    stream = torch.cuda.current_stream()
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    ev_part = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    ev_app = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]

    local = dec.local if group else dec

    def step(i=None):
        if st["kv_new"] is not None:
            if i is not None:
                ev_app[i][0].record(stream)
            dec.append(st["kv_new"], st["pos"], st["req"], st["bt"])
            if i is not None:
                ev_app[i][1].record(stream)
        if i is not None:
            ev_part[i][0].record(stream)
        local.partial(st["q"], st["bt"], st["seq_lens"])
        if i is not None:
            ev_part[i][1].record(stream)
        if group:
            dec.xchg.exchange(local.o_part, local.lse_part)
        else:
            dec.merge()

    for _ in range(args.warmup):
        step()
    barrier(dist)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)                       # let the sampler take its first reading
    barrier(dist)
    launches0 = dcp.dcp_launch_count()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()           # bounds an `ncu --profile-from-start off` launch list
    clocks.mark()
    t0.record(stream)
    for i in range(args.steps):
        ev_step[i][0].record(stream)
        step(i)
        ev_step[i][1].record(stream)
    t1.record(stream)
    barrier(dist)
    clocks.mark()
    torch.cuda.profiler.stop()
    launches = dcp.dcp_launch_count() - launches0
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    part_ms = [a.elapsed_time(b) for a, b in ev_part]
    if dec.status_bits() != 0:
        raise RuntimeError(f"device status {dec.status_bits()} after the timed steps")
    ms_per_step = max_over_ranks(dist, total_ms / args.steps)
    part_ms_avg = max_over_ranks(dist, sum(part_ms) / len(part_ms))
    append = None
    if st["kv_new"] is not None:
        # the owner-filtered append of the step's new rows, on its own: each row is
        # read once (1152 B + its position and request) and written once by its owner
        app_ms = max_over_ranks(dist, statistics.mean(a.elapsed_time(b) for a, b in ev_app))
        rows = st["kv_new"].shape[0]
        append = {"rows": rows, "us": round(app_ms * 1e3, 2),
                  "note": "dcp_kv_append alone (CUDA events around it inside the timed steps)"}
        if not group:
            app_bytes = rows * (2 * KV_ROW_BYTES + 12)
            append.update({"bytes": app_bytes, "GB/s": round(app_bytes / (app_ms * 1e-3) / 1e9, 1)})

    # end-to-end through the public API with host buffers (H2D inputs, D2H result each step)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, cfg, st, dist, acct)

    peaks = load_peaks()
    # the whole job's KV per step (all shards on all ranks) over the step time
    kv_gbs = acct["kv_bytes"] / (ms_per_step * 1e-3) / 1e9
    t_hbm = acct["bytes_alg"] / (peaks["hbm_gbs"] * 1e9 * world)
    t_tc = acct["flops_alg"] / (peaks["bf16_tflops"] * 1e12 * world)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    partial_achieved = acct["partial_bytes_alg"] / (part_ms_avg * 1e-3) / 1e9
    part_flops = acct.get("flops_alg_rank", acct["flops_alg"]) / (part_ms_avg * 1e-3) / 1e12
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(partial_achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(partial_achieved / peaks["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(part_flops, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(part_flops / peaks["bf16_tflops"], 4)}
    # the committed captures are of the default launch (full batch, fp32 partials)
    roof["traffic"] = recorded_traffic(cfg.name) if args.batch is None and args.partials == "fp32" else None
    roof["kernel"] = "dcp_mla_decode_partial (all its launches, CUDA events on the launching stream)"
    roof["peak_source"] = f"{peaks['source']} MEASURED_PEAKS.json" if peaks["source"] == "measured" else "fallback"
    if group:
        roof["kernel"] = ("dcp_mla_decode_partial of this rank's shards (all its launches, CUDA events on the "
                          "launching stream; max over ranks)")
        roof["traffic"] = None
    result = {
        "metric": METRIC,
        "value": round(kv_gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "roofline_frac_step": round(max(t_hbm, t_tc) / (ms_per_step * 1e-3), 4),
        "step_binding_roofline": bound,
        "higher_is_better": True,
        "scaling": "strong" if group else "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 latent rows and queries, shuffled block table)",
        "config": config_dict(cfg, st["S"], world, args.exchange if group else None, args.partials),
        "roofline": roof,
        "partial_ms": round(part_ms_avg, 5),
        "append": append,
        "step_ms_median": round(statistics.median(step_ms), 5),
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": clk,
    }
    if group:
        result["exchange"] = {"strategy": args.exchange, "collectives": "NCCL (torch.distributed)",
                              "bytes_per_rank_per_step": dec.xchg.bytes_sent(),
                              "shards_per_gpu": dec.local.shard_end - dec.local.shard_begin,
                              "heads_per_gpu": dec.head_end - dec.head_begin}
    return result


RELAYOUT_METRIC = "prefill-to-decode relayout: moved KV GB/s (read + write), % of HBM roofline"
RELAYOUT_SRC_PAGE = 64   # rows per page of the prefill-side pool


def run_relayout_op(args, cfg, rank, world, dist, device):
    """Timed dcp_kv_relayout: every token of the workload's requests, prefilled
    without context sharding into a paged pool (pages of 64 rows, shuffled), is
    moved into its owner's compact pool (all N shards on this GPU)."""
    import context_sharded_mla_gb300 as dcp
    lay = dcp.Layout(cfg.N, cfg.I, cfg.P)
    S = workloads.lengths(cfg)
    g = torch.Generator(device=device).manual_seed(17)
    Ps = RELAYOUT_SRC_PAGE
    src_pages = [(int(x) + Ps - 1) // Ps for x in S]
    total_src = sum(src_pages)
    perm = torch.randperm(total_src, generator=g, device=device).to(torch.int32)
    src_bt = torch.full((cfg.B, max(src_pages)), -1, dtype=torch.int32, device=device)
    k = 0
    for b in range(cfg.B):
        src_bt[b, :src_pages[b]] = perm[k:k + src_pages[b]]
        k += src_pages[b]
    src_pool = torch.empty(total_src * Ps, 576, dtype=torch.bfloat16, device=device).normal_(generator=g)
    bt, pool_pages = workloads.block_table(cfg, S)
    bt = bt.to(device)
    arena = torch.zeros(cfg.N, pool_pages * cfg.P, 576, dtype=torch.bfloat16, device=device)
    pos = torch.cat([torch.arange(int(x), dtype=torch.int64, device=device) for x in S])
    req = torch.cat([torch.full((int(x),), b, dtype=torch.int32, device=device) for b, x in enumerate(S)])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    T = pos.numel()
    bytes_alg = T * (2 * 1152 + 12)           # read + write of each latent row, its position and request
    stream = torch.cuda.current_stream()

    def call(p_, r_):
        dcp.dcp_kv_relayout(lay, 0, cfg.N, src_pool, Ps, src_bt, src_bt.shape[1], p_, r_, bt, bt.shape[1], arena,
                            pool_pages, status)

    for _ in range(args.warmup):
        call(pos, req)
    barrier(dist)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    launches0 = dcp.dcp_launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()
    clocks.mark()
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        call(pos, req)
        ev[i][1].record(stream)
    t1.record(stream)
    barrier(dist)
    clocks.mark()
    torch.cuda.profiler.stop()
    launches = dcp.dcp_launch_count() - launches0
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed relayouts")
    ms = max_over_ranks(dist, t0.elapsed_time(t1) / args.steps)
    kernel_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    peaks = load_peaks()
    achieved = bytes_alg / (kernel_ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        pos_h, req_h = pos.cpu().pin_memory(), req.cpu().pin_memory()
        st_h = torch.empty(1, dtype=torch.int32).pin_memory()
        pos_d, req_d = torch.empty_like(pos), torch.empty_like(req)

        def e2e_step():
            pos_d.copy_(pos_h, non_blocking=True)
            req_d.copy_(req_h, non_blocking=True)
            call(pos_d, req_d)
            st_h.copy_(status, non_blocking=True)

        for _ in range(3):
            e2e_step()
        n = max(1, min(args.steps, 50))
        a_ = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(n):
            e2e_step()
        b_.record(stream)
        torch.cuda.synchronize()
        e_ms = a_.elapsed_time(b_) / n
        e2e = {"value": round(bytes_alg / (e_ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s", "ms_per_step": round(e_ms, 5),
               "h2d_bytes_per_step": T * 12, "d2h_bytes_per_step": 4, "steps": n,
               "path": "dcp_kv_relayout over the C ABI; token list copied from pinned host memory each step"}
    return {
        "metric": RELAYOUT_METRIC, "value": round(bytes_alg / (ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 latent rows, shuffled source and destination page tables)",
        "config": relayout_config(cfg),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "kernel": "kv_relayout_kernel (CUDA events on the launching stream)",
                     "peak_source": f"{peaks['source']} MEASURED_PEAKS.json" if peaks["source"] == "measured"
                     else "fallback"},
        "gpu_launches": launches, "e2e": e2e, "clocks": clk,
    }


def time_oracle_relayout(cfg, budget_s):
    """The oracle's pd_relayout on a bounded sample: positions of one request of the same layout."""
    import numpy as np
    from oracle import layout as olayout
    Ps = RELAYOUT_SRC_PAGE
    rng = np.random.default_rng(5)
    L = 65536
    src_bt = rng.permutation(L // Ps)[None, :]
    src = rng.integers(0, 65535, size=(L, 576), dtype=np.uint16)
    rows = int(olayout.count(0, L, cfg.N, cfg.I)) + cfg.I
    dpages = (rows + cfg.P - 1) // cfg.P
    bt = rng.permutation(dpages)[None, :]
    arena = np.zeros((cfg.N, dpages * cfg.P, 576), dtype=np.uint16)
    pos = np.arange(L)
    done, t0 = 0, time.time()
    while done == 0 or time.time() - t0 < budget_s:  # whole passes over the request
        olayout.pd_relayout(arena, src, src_bt, Ps, pos, np.zeros_like(pos), bt, cfg.N, cfg.I, cfg.P)
        done += L
    secs = time.time() - t0
    return done * (2 * 1152 + 12), secs, (f"{done // L} pass(es) over one {L}-token request, same layout, "
                                          "python/numpy, one thread")


ABSORB_METRIC = "absorption products (q_nope @ w_kc, o @ w_vc): moved GB/s, % of HBM roofline"
L2_FLUSH_BYTES = 256 << 20      # written between timed steps: twice the 129 MB L2


def absorb_bytes(T, H, o_bytes_per_el=2, v_bytes_per_el=2):
    """Algorithmic bytes of one pass of each product: (query side, output side)."""
    q_side = T * H * (128 + 64) * 2 + H * 128 * 512 * 2 + T * H * 576 * 2
    o_side = T * H * 512 * o_bytes_per_el + H * 512 * 128 * 2 + T * H * 128 * v_bytes_per_el
    return q_side, o_side


def run_absorb_op(args, cfg, rank, world, dist, device):
    """Timed dcp_absorb_q + dcp_absorb_o at the workload's decode shapes (T = B x q_len
    query tokens, H heads; synthetic bf16 weights; o in the merge's output dtype)."""
    import context_sharded_mla_gb300 as dcp
    T, H = cfg.B * cfg.q_len, cfg.H
    qp = workloads.gen_q_proj(cfg, device)
    w_kc, w_vc = (w.to(device) for w in workloads.gen_absorb_weights(cfg, device))
    o_dtype = torch.float32 if cfg.out_dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device).manual_seed(23)
    o = torch.randn(cfg.B, cfg.q_len, H, 512, generator=g, device=device).to(o_dtype)
    q = torch.empty(cfg.B, cfg.q_len, H, 576, dtype=torch.bfloat16, device=device)
    v = torch.empty(cfg.B, cfg.q_len, H, 128, dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    # the decode step's partials at these shapes (f32, N parts), for the merge and
    # the fused merge + output product
    o_part = torch.randn(cfg.N, T, H, 512, generator=g, device=device)
    lse_part = torch.randn(cfg.N, T, H, generator=g, device=device)
    o_merged = torch.empty(T, H, 512, dtype=o_dtype, device=device)
    lse_merged = torch.empty(T, H, dtype=torch.float32, device=device)
    base = dcp.DCP_LSE_BASE_2 if cfg.base == 2 else dcp.DCP_LSE_BASE_E
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_sum = torch.empty((), dtype=torch.float32, device=device)
    q_bytes, o_bytes = absorb_bytes(T, H, o.element_size(), 2)

    def flush_l2():
        # write a buffer twice the L2, then read it back: the next step starts
        # with its inputs out of L2 and no dirty lines left to write back
        flush.zero_()
        torch.sum(flush, dim=0, out=flush_sum)
    stream = torch.cuda.current_stream()

    def call(qp_, o_):
        dcp.dcp_absorb_q(qp_[..., :128], qp_[..., 128:], w_kc, q, status)
        dcp.dcp_absorb_o(o_, w_vc, v, status)

    for _ in range(args.warmup):
        flush_l2()
        call(qp, o)
    barrier(dist)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    launches0 = dcp.dcp_launch_count()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    torch.cuda.profiler.start()
    clocks.mark()
    # The kernels take microseconds, less than the host needs to submit them:
    # a spin of a few ms first lets the host queue the steps ahead of the GPU,
    # so the events time the kernels, not the host.
    torch.cuda._sleep(20_000_000)
    for i in range(args.steps):
        flush_l2()                         # L2 cold for every step (outside the kernel events)
        ev[i][0].record(stream)
        dcp.dcp_absorb_q(qp[..., :128], qp[..., 128:], w_kc, q, status)
        ev[i][1].record(stream)
        dcp.dcp_absorb_o(o, w_vc, v, status)
        ev[i][2].record(stream)
        flush_l2()
        ev[i][3].record(stream)
        dcp.dcp_lse_merge(o_part.view(cfg.N, -1, 512), lse_part.view(cfg.N, -1), base, o_merged.view(-1, 512),
                          lse_merged.view(-1))
        ev[i][4].record(stream)
        flush_l2()
        ev[i][5].record(stream)
        dcp.dcp_lse_merge_absorb_o(o_part, lse_part, base, w_vc, v.view(T, H, 128), lse_merged, status)
        ev[i][6].record(stream)
    barrier(dist)
    clocks.mark()
    torch.cuda.profiler.stop()
    launches = dcp.dcp_launch_count() - launches0
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed absorption products")
    q_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    o_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    merge_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in ev)
    fused = [e[5].elapsed_time(e[6]) for e in ev]
    ms = max_over_ranks(dist, q_ms + o_ms)
    peaks = load_peaks()
    dom = ("absorb_kernel (query side)", q_bytes, q_ms) if q_ms >= o_ms else ("absorb_kernel (output side)",
                                                                              o_bytes, o_ms)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        qp_h = qp.cpu().pin_memory()
        o_h = o.cpu().pin_memory()
        q_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        v_h = torch.empty(v.shape, dtype=v.dtype).pin_memory()
        qp_d, o_d = torch.empty_like(qp), torch.empty_like(o)

        def e2e_step():
            qp_d.copy_(qp_h, non_blocking=True)
            o_d.copy_(o_h, non_blocking=True)
            call(qp_d, o_d)
            q_h.copy_(q, non_blocking=True)
            v_h.copy_(v, non_blocking=True)

        for _ in range(3):
            e2e_step()
        n = max(1, min(args.steps, 200))
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(n):
            e2e_step()
        b_.record(stream)
        torch.cuda.synchronize()
        e_ms = a_.elapsed_time(b_) / n
        e2e = {"value": round((q_bytes + o_bytes) / (e_ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 5),
               "h2d_bytes_per_step": qp.numel() * 2 + o.numel() * o.element_size(),
               "d2h_bytes_per_step": q.numel() * 2 + v.numel() * 2, "steps": n,
               "path": "dcp_absorb_q + dcp_absorb_o over the C ABI; q_proj and o copied from pinned host memory, "
                       "q and v copied back, every step (weights resident)"}
    return {
        "metric": ABSORB_METRIC, "value": round((q_bytes + o_bytes) / (ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "us_per_step": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) query projection and o; weights N(0, 1/fan_in), bf16)",
        "config": absorb_config(cfg),
        "kernels_us": {"absorb_q": round(q_ms * 1e3, 3), "absorb_o": round(o_ms * 1e3, 3),
                       "lse_merge": round(merge_ms * 1e3, 3),
                       "lse_merge_absorb_o": round(statistics.mean(fused) * 1e3, 3)},
        "products_step_cost_us": {
            "separate": round((q_ms + o_ms) * 1e3, 3),
            "fused": round((q_ms + statistics.mean(fused) - merge_ms) * 1e3, 3),
            "note": "what the two products add to a decode step: absorb_q + absorb_o after a separate merge, or "
                    "absorb_q + (fused merge-and-product - plain merge); N f32 partials, L2 flushed before each call"},
        "bytes_alg": {"absorb_q": q_bytes, "absorb_o": o_bytes},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": (recorded_traffic("absorb_q") if q_ms >= o_ms and cfg.name == "k3"
                                 and args.batch is None else None),
                     "kernel": f"{dom[0]} (CUDA events on the launching stream)",
                     "peak_source": f"{peaks['source']} MEASURED_PEAKS.json" if peaks["source"] == "measured"
                     else "fallback"},
        "gpu_launches": launches, "e2e": e2e, "clocks": clk,
    }


def time_oracle_absorb(cfg, budget_s):
    """The oracle's absorb_q + absorb_o on a bounded sample: all T tokens, a slice of the heads per pass."""
    import numpy as np
    from oracle import absorb as oabsorb
    T, H = cfg.B * cfg.q_len, cfg.H
    qp = workloads.gen_q_proj(cfg).reshape(T, H, 192).to(torch.float64).numpy()
    w_kc, w_vc = (w.to(torch.float64).numpy() for w in workloads.gen_absorb_weights(cfg))
    o = np.random.default_rng(23).standard_normal((T, H, 512))
    hs = max(1, min(H, 8))
    q_bytes, o_bytes = absorb_bytes(T, H, 2, 2)
    done, t0 = 0, time.time()
    while done == 0 or time.time() - t0 < budget_s:
        h0 = (done * hs) % H
        sl = slice(h0, min(H, h0 + hs))
        oabsorb.absorbed_query(qp[:, sl, :128], qp[:, sl, 128:], w_kc[sl])
        oabsorb.absorb_o(o[:, sl], w_vc[sl])
        done += 1
    secs = time.time() - t0
    heads = done * hs
    return (q_bytes + o_bytes) * heads / H, secs, (f"{done} passes of {hs} of {H} heads x {T} tokens (both "
                                                    f"products, fp64 numpy einsum); throughput counts that share "
                                                    f"of the algorithmic bytes")


def run_e2e(args, cfg, st, dist, acct):
    """The same step end to end through the decoder's public calls, with every
    step's inputs copied from pinned host memory and its merged output read back.

    Copies run on a second stream, as a serving loop would run them: the inputs
    of step i + 1 (double-buffered on the device) go up while step i computes,
    and step i's output comes back while step i + 1's partials run; only step
    i + 1's merge, which rewrites the output buffer, waits for that read.  Every
    byte is still copied every step inside the timed region."""
    dec = st["dec"]
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    group = hasattr(dec, "xchg")            # a DCP group rank: its output is its heads' slice
    local = dec.local if group else dec
    o_out, lse_out = (dec.xchg.o, dec.xchg.lse) if group else (dec.o, dec.lse)
    has_new = st["kv_new"] is not None
    names = ["q", "seq_lens"] + (["kv_new", "pos", "req"] if has_new else [])
    src = {"q": st["q"], "seq_lens": st["seq_lens"]}
    if has_new:
        src.update(kv_new=st["kv_new"], pos=st["pos"], req=st["req"])
    host = {n: src[n].cpu().pin_memory() for n in names}
    dev = [{n: torch.empty_like(src[n]) for n in names} for _ in range(2)]
    o_host = [torch.empty(o_out.shape, dtype=o_out.dtype).pin_memory() for _ in range(2)]
    lse_host = [torch.empty(lse_out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_host[0].numel() * o_host[0].element_size() + lse_host[0].numel() * 4
    up = [torch.cuda.Event() for _ in range(2)]      # inputs of the step using buffer k are on the device
    used = [torch.cuda.Event() for _ in range(2)]    # the step using buffer k has read its inputs
    done = [torch.cuda.Event() for _ in range(2)]    # the step's output is complete
    back = [torch.cuda.Event() for _ in range(2)]    # the step's output is on the host
    state = {"read": None}

    def upload(k):
        copy.wait_event(used[k])                     # the step two back has finished with buffer k
        with torch.cuda.stream(copy):
            for n in names:
                dev[k][n].copy_(host[n], non_blocking=True)
        up[k].record(copy)

    def step(i):
        k = i & 1
        d = dev[k]
        main.wait_event(up[k])
        if has_new:
            dec.append(d["kv_new"], d["pos"], d["req"], st["bt"])
        local.partial(d["q"], st["bt"], d["seq_lens"])
        used[k].record(main)
        upload(k ^ 1)                                # the next step's inputs go up now
        if state["read"] is not None:
            main.wait_event(state["read"])           # the previous output has been read back
        if group:
            dec.xchg.exchange(local.o_part, local.lse_part)
        else:
            dec.merge()
        done[k].record(main)
        copy.wait_event(done[k])
        with torch.cuda.stream(copy):
            o_host[k].copy_(o_out.reshape(o_host[k].shape), non_blocking=True)
            lse_host[k].copy_(lse_out.reshape(lse_host[k].shape), non_blocking=True)
        back[k].record(copy)
        state["read"] = back[k]

    for k in range(2):
        used[k].record(main)
    upload(0)
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    barrier(dist)
    n = max(1, min(args.steps, 200))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w = max(3, args.warmup)
    # the timed region starts before the first timed step's inputs go up
    t0.record(main)
    copy.wait_event(t0)
    for i in range(w, w + n):
        step(i)
    main.wait_event(state["read"])                   # the last output is on the host
    t1.record(main)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, t0.elapsed_time(t1) / n)
    path = ("DcpGroupDecoder over the C ABI and NCCL (query replicated to every rank, each rank reads back "
            "its heads' o / lse), pinned host buffers" if group else
            "ShardedMlaDecoder append / partial / merge over the C ABI, pinned host buffers")
    return {"value": round(acct["kv_bytes"] / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "path": path,
            "overlap": "inputs of step i+1 copied up, and step i's output read back, on a second stream while "
                       "the device computes; every copy runs every step inside the timed region"}


def recorded_traffic(key):
    """DRAM bytes per launch of a kernel from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        import hashlib
        entry = rec.get(key)
        if not entry:
            return None
        src = os.path.join(ROOT, entry.get("source", "context_sharded_mla_gb300/csrc/dcp_decode.cu"))
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if entry.get("source_sha") != h:
            return None
        scale = entry.get("scale_to_full", 1.0)
        return int(entry["dram_bytes_per_launch"] * scale)
    except (OSError, ValueError, KeyError):
        return None


def config_dict(cfg, S, world, strategy=None, partials="fp32"):
    """The decode step's `config`, from the workload alone (both arms print the same one)."""
    d = {"workload": workloads.DESCRIPTIONS[cfg.name] if cfg.name in workloads.DESCRIPTIONS else cfg.name,
         "B": cfg.B, "H": cfg.H, "q_len": cfg.q_len, "S_total": int(S.sum()), "S_max": int(S.max()),
         "n_shards": cfg.N, "interleave": cfg.I, "page_size": cfg.P, "lse_base": "2" if cfg.base == 2 else "e",
         "new_tokens_per_request": max(cfg.append, cfg.chunk), "out_dtype": cfg.out_dtype,
         "partials": partials, "global_batch": cfg.B, "seq_len": int(S.max()),
         "parallelism": ("1 GPU holds all N shards" if strategy is None else
                         f"DCP over {world} GPUs: {cfg.N // world} shards and {cfg.H // world} output heads per GPU, "
                         f"query replicated, {strategy} exchange of the partials"),
         "l2": f"inputs larger than L2 ({int(S.sum()) * KV_ROW_BYTES / 1e9:.2f} GB of KV per step), no flush"}
    return d


def relayout_config(cfg):
    S = workloads.lengths(cfg)
    Ps = RELAYOUT_SRC_PAGE
    return {"workload": f"relayout of {workloads.DESCRIPTIONS.get(cfg.name, cfg.name)} requests, prefilled "
                        f"without context sharding (source pages of {Ps} rows), into all {cfg.N} shards",
            "B": cfg.B, "tokens": int(S.sum()), "n_shards": cfg.N, "interleave": cfg.I, "page_size": cfg.P,
            "source_page_size": Ps, "l2": "source and destination far larger than L2, no flush"}


def absorb_config(cfg):
    T, H = cfg.B * cfg.q_len, cfg.H
    o_dtype = "float32" if cfg.out_dtype == "f32" else "bfloat16"
    return {"workload": f"absorption products at the decode shapes of "
                        f"{workloads.DESCRIPTIONS.get(cfg.name, cfg.name)}: T={T} query tokens, H={H}, "
                        f"w_kc [H,128,512], w_vc [H,512,128], o {o_dtype}, v bf16",
            "T": T, "H": H, "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MB written and "
                                   "read back, outside the timed kernels)"}


# ----------------------------------------------------------------------------- oracle (CPU) arm

def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info()]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def time_oracle(cfg, budget_s, min_units=1, device=None):
    """Time the fp64 oracle on whole-request units (all heads, all shards + merge) of cfg.

    Inputs are the same seeded rows (drawn on `device`, copied to the host
    before the clock starts).  Returns (kv_bytes_processed, seconds, sample description).
    """
    import numpy as np
    from oracle import attention
    S = workloads.lengths(cfg)
    gen_dev = device or "cpu"
    q = workloads.gen_q(cfg, gen_dev).cpu()
    order = sorted(range(cfg.B), key=lambda b: int(S[b]))
    done_bytes, elapsed, used = 0, 0.0, []
    heads_all = cfg.H
    for b in order:
        kv = workloads.gen_kv(cfg, b, int(S[b]), gen_dev).cpu().to(torch.float64).numpy()
        qb = q[b].to(torch.float64).numpy()
        t0 = time.perf_counter()
        attention.sharded_attention(qb, kv, int(S[b]), cfg.N, cfg.I, workloads.SCALE, cfg.base)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_bytes += int(S[b]) * KV_ROW_BYTES
        used.append(b)
        del kv
        if len(used) >= min_units and elapsed >= budget_s:
            break
    desc = (f"{len(used)} whole request(s) of {cfg.B} ({sum(int(S[b]) for b in used)} tokens, all {heads_all} "
            f"heads, all {cfg.N} shards + merge), fp64 numpy")
    return done_bytes, elapsed, desc


def time_oracle_fraction(cfg, seconds_target, device=None):
    """One bounded oracle step: request 0 restricted to enough heads to take ~seconds_target."""
    import numpy as np
    from oracle import attention
    S = workloads.lengths(cfg)
    gen_dev = device or "cpu"
    b = int(torch.argmin(S))
    q = workloads.gen_q(cfg, gen_dev)[b].cpu().to(torch.float64).numpy()
    kv = workloads.gen_kv(cfg, b, int(S[b]), gen_dev).cpu().to(torch.float64).numpy()
    # calibrate on one head
    t0 = time.perf_counter()
    attention.sharded_attention(q[:, :1], kv, int(S[b]), cfg.N, cfg.I, workloads.SCALE, cfg.base)
    t1 = time.perf_counter() - t0
    heads = int(max(1, min(cfg.H, seconds_target / max(t1, 1e-6))))
    return b, q, kv, heads, int(S[b])


def run_reference(args, cfg, rank, world):
    """Times the oracle (the reference arm for this build) on a bounded sample per step."""
    from oracle import attention
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    budget_per_step = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    b, q, kv, heads, S_b = time_oracle_fraction(cfg, budget_per_step, dev)
    for _ in range(args.warmup):
        attention.sharded_attention(q[:, :heads], kv, S_b, cfg.N, cfg.I, workloads.SCALE, cfg.base)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attention.sharded_attention(q[:, :heads], kv, S_b, cfg.N, cfg.I, workloads.SCALE, cfg.base)
    dt = (time.perf_counter() - t0) / args.steps
    eq_bytes = S_b * KV_ROW_BYTES * heads / cfg.H      # the share of the request's work done per step
    value = eq_bytes / dt / 1e9
    cores = oracle_threads()
    sample = (f"per step: request {b} ({S_b} tokens), {heads} of {cfg.H} heads, all {cfg.N} shards + merge "
              f"(fp64 numpy oracle); throughput counts {heads}/{cfg.H} of that request's KV bytes")
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "strong" if world > 1 or args.group else "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": config_dict(cfg, workloads.lengths(cfg), world, args.exchange if world > 1 or args.group else None,
                              args.partials),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_op(args, cfg, rank, world):
    """--impl reference for --op relayout / absorb: the oracle of that op, timed per step on a bounded sample."""
    if rank != 0:
        return None
    metric, time_op = ((RELAYOUT_METRIC, time_oracle_relayout) if args.op == "relayout"
                       else (ABSORB_METRIC, time_oracle_absorb))
    budget = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_op(cfg, budget)
    nbytes, secs = 0.0, 0.0
    for _ in range(args.steps):
        b_, s_, desc = time_op(cfg, budget)
        nbytes, secs = nbytes + b_, secs + s_
    value = nbytes / secs / 1e9
    return {
        "metric": metric, "impl": "reference", "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": relayout_config(cfg) if args.op == "relayout" else absorb_config(cfg),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="k3", choices=sorted(workloads.DESCRIPTIONS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller case for profiling)")
    ap.add_argument("--partials", default="fp32", choices=["fp32", "bf16"],
                    help="dtype of the per-shard partial outputs o_r (fp32 by default; bf16 is the all-to-all "
                         "wire format of the pages)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--group", action="store_true",
                    help="run the multi-GPU (DCP group) step even with --gpus 1: the exchange kernels run, the "
                         "collectives are skipped")
    ap.add_argument("--exchange", default="a2a", choices=["a2a", "ag_rs"],
                    help="with --gpus N > 1: all-to-all of the packed partials (default) or AllGather(lse) + "
                         "ReduceScatter")
    ap.add_argument("--op", default="decode", choices=["decode", "relayout", "absorb"],
                    help="decode: the decode step (default); relayout: the prefill-to-decode relayout; "
                         "absorb: the two absorption products")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_info()
    cfg = workloads.config(args.workload)
    if args.batch:
        cfg = workloads.config(args.workload, B=args.batch)
    if args.impl == "reference":
        out = (run_reference(args, cfg, rank, world) if args.op == "decode"
               else run_reference_op(args, cfg, rank, world))
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")   # plain NVLink transfers, no multicast objects
    dist = init_dist(world, "nccl")
    if args.op in ("relayout", "absorb"):
        run_op, time_op = ((run_relayout_op, time_oracle_relayout) if args.op == "relayout"
                           else (run_absorb_op, time_oracle_absorb))
        result = run_op(args, cfg, rank, world, dist, device)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            nbytes, secs, desc = time_op(cfg, args.cpu_budget)
            result["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 6), "unit": "GB/s", "cores": 1,
                                      "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        if rank == 0:
            print(json.dumps(result), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0
    result = run_ours(args, cfg, rank, world, dist, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kv_bytes, secs, desc = time_oracle(cfg, args.cpu_budget, device=device)
        result["cpu_baseline"] = {"value": round(kv_bytes / secs / 1e9, 6), "unit": "GB/s",
                                  "cores": oracle_threads(), "kind": "oracle", "sample": desc,
                                  "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
