"""Benchmark of the tree-verification hot path on GB300 over one batch of the
Mamba-2-like workload (B=16 requests, H=24 heads, dk=128, dv=64, 16-node top-4
draft trees, bf16 q/k/v, fp32 states, scalar decay).  One step verifies the
tree, runs the greedy acceptance walk and commits the accepted path:

  --pipeline one (default): tv_accept_commit_verify, one launch: the greedy walk
      of the previous tree, the commit of its path to the state in place, and the
      verification of the current tree against the committed state.  Every step
      does one walk, one commit and one verification; the state stays resident and
      is streamed once.
  --pipeline fused: tv_commit_verify (the previous step's accepted paths applied
      to the state in place, then the tree verified against it) + tv_accept_greedy.
  --pipeline separate: tv_verify + tv_accept_commit (walk and commit in one
      launch), the state streamed by both kernels.

Prints one JSON line (rank 0).  Metric: tree-verify node-head updates per
second (node-heads = nodes x heads per batch), whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: inputs resident in HBM; R distinct input sets (> 4x L2 in total) are
used in rotation so every step reads cold data; the K timed steps run as CUDA
graph replays bracketed by CUDA events on the launching stream, with a barrier
and synchronize on both sides, max over ranks.  `e2e` repeats the step through
the Python binding with pinned host buffers and the host<->device copies inside
the timed region.  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify node-head updates/s"
UNIT = "node-head/s"
WORKLOADS = {
    1: "single request, 1 head, dk=dv=16, fp32 q/k/v, 8-node random tree, scalar decay",
    2: ("Mamba-2-like layer: B=16 requests, H=24 heads, dk=128, dv=64, 16-node top-4 draft "
        "tree (4 chains of depth 4), bf16 q/k/v, fp32 H0, scalar decay"),
    3: ("GLA-like layer: B=32, H=16, dk=dv=128, bf16 q/k/v, fp32 H0, per-channel decay, "
        "64-node best-first trees (depth <= 8, Dirichlet(0.3))"),
    4: ("mixed-budget batch: B=128, H=32, dk=dv=128, bf16 q/k/v, fp32 H0, scalar decay, "
        "tree sizes in {4..128}, depth cap 12"),
    5: ("large-tree stack: B=8, 36 layers x 32 heads (H=1152), dk=dv=128, bf16 q/k/v, fp32 H0, "
        "per-channel decay, 256-node best-first trees (depth <= 16, Dirichlet(0.2))"),
}
WORKLOAD = WORKLOADS[2]
_CS = "tree_speculative_verify_tv_gb300/csrc/"
# sources behind each kernel whose DRAM traffic was captured with ncu
TRAFFIC_SOURCES = {
    "verify": [_CS + f for f in ("verify_tc_fused.cu", "tc_common.cuh", "tc_ptx.cuh",
                                 "tv_internal.cuh", "greedy_walk.cuh")],
    "commit_verify": [_CS + f for f in ("verify_tc_fused.cu", "tc_common.cuh", "tc_ptx.cuh",
                                        "tv_internal.cuh", "greedy_walk.cuh")],
    "accept_commit_verify": [_CS + f for f in ("verify_tc_fused.cu", "tc_common.cuh",
                                               "tc_ptx.cuh", "tv_internal.cuh",
                                               "greedy_walk.cuh")],
    "tree_attention": [_CS + f for f in ("tree_attention.cu", "tc_common.cuh", "tc_ptx.cuh",
                                         "tv_internal.cuh")],
}
KERNEL_NAMES = {1: "simt", 2: "tcgen05 one unit per CTA",
                3: "tcgen05 fused (decay in the factors; up to 256-node per-channel trees: "
                   "context on tensor cores, tree term by fp32 walks)",
                4: "tcgen05 large trees (staged or node tiles)"}


DEFAULT_STEPS = {1: 40000, 2: 40000, 3: 5000, 4: 400, 5: 40}
DEFAULT_WARMUP = {1: 200, 2: 200, 3: 50, 4: 10, 5: 3}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 40000 for config 2, fewer for the larger configs)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sets", type=int, default=0, help="rotated input sets (0 = auto, >4x L2)")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--variant", type=int, default=0, help="tv_verify variant (0 auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration block (every configuration's tv_verify "
                         "at full size)")
    ap.add_argument("--fold", type=int, default=32,
                    help="also time one verify launch over this many config-2 layers folded "
                         "into the head axis (0 = skip)")
    ap.add_argument("--profile-folded", type=int, default=None, metavar="VARIANT",
                    help="profiling aid: only run 3 verify launches of this tv_variant over "
                         "--fold config-2 layers folded into the head axis, then exit")
    ap.add_argument("--pipeline", default="one", choices=["one", "fused", "separate"],
                    help="step as tv_accept_commit_verify (one), as tv_commit_verify + "
                         "tv_accept_greedy (fused) or as tv_verify + tv_accept_commit "
                         "(separate)")
    ap.add_argument("--attention-ctx", type=int, default=4096,
                    help="shared-prefix positions per request for the tree-attention line "
                         "(0 = skip it)")
    ap.add_argument("--profile-verify", type=int, default=None, metavar="VARIANT",
                    help="profiling aid: only run 3 verify launches of this tv_variant on "
                         "--config's workload (config 5 as 2 layers of 32 heads, 512 units), "
                         "then exit")
    ap.add_argument("--profile-extras", action="store_true",
                    help="three launches each of tv_build_tree and tv_accept_stochastic (ncu)")
    ap.add_argument("--profile-attention", action="store_true",
                    help="profiling aid: only run 3 tree-attention launches of the attention "
                         "workload, then exit")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5],
                    help="workload (default 2: the configuration the HBM target is quoted on)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.config]
    if args.warmup is None:
        args.warmup = DEFAULT_WARMUP[args.config]
    return args


# ---------------------------------------------------------------- byte accounting


def verify_bytes(b) -> int:
    """Algorithmic HBM bytes of one tv_verify launch: H0 read once, every factor
    row read once, every output row written once, tree metadata read once."""
    qk = 2 if b.qkv_dtype == "bf16" else 4
    g = 4 if b.decay == "scalar" else 4 * b.dk
    per_node_head = 2 * b.dk * qk + b.dv * qk + g + 4 * b.dv
    return (b.B * b.H * 4 * b.dk * b.dv + b.T * b.H * per_node_head + 8 * b.T
            + 4 * (b.B + 1))


def verify_bytes_of(d) -> int:
    """verify_bytes for a DeviceBatch."""
    qk = 2 if d.qkv_dtype == 0 else 4
    g = 4 if d.decay == 0 else 4 * d.dk
    per_node_head = 2 * d.dk * qk + d.dv * qk + g + 4 * d.dv
    return d.B * d.H * 4 * d.dk * d.dv + d.T * d.H * per_node_head + 8 * d.T + 4 * (d.B + 1)


def commit_verify_bytes(b, lens) -> int:
    """Algorithmic HBM bytes of one tv_commit_verify launch: those of tv_verify, the
    committed state rows written back (requests with a non-empty path), and the
    path's factor rows, offsets, lengths and paths."""
    qk = 2 if b.qkv_dtype == "bf16" else 4
    g = 4 if b.decay == "scalar" else 4 * b.dk
    lens = np.asarray(lens)
    written = int(np.count_nonzero(lens)) * b.H * 4 * b.dk * b.dv
    L = int(np.sum(lens))
    return (verify_bytes(b) + written + L * b.H * (b.dk * qk + b.dv * qk + g) + 4 * L
            + 4 * (b.B + 1) + 4 * b.B + 4 * b.B * b.max_depth)


def accept_commit_verify_bytes(b, lens) -> int:
    """Algorithmic HBM bytes of one tv_accept_commit_verify launch: those of
    tv_commit_verify, plus the previous tree's parents, draft and target tokens and
    root tokens the walk reads and the bonus tokens it writes."""
    return commit_verify_bytes(b, lens) + 12 * b.T + 4 * b.B + 4 * b.B


def commit_bytes(b, lens) -> int:
    """H0 read + H_new written, plus the accepted path's factor rows."""
    qk = 2 if b.qkv_dtype == "bf16" else 4
    g = 4 if b.decay == "scalar" else 4 * b.dk
    L = int(np.sum(lens))
    return b.B * b.H * 8 * b.dk * b.dv + L * b.H * (b.dk * qk + b.dv * qk + g)


def kernel_source_hash(name: str) -> str:
    h = hashlib.sha256()
    for p in TRAFFIC_SOURCES[name]:
        fp = os.path.join(ROOT, p)
        if os.path.exists(fp):
            h.update(open(fp, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """Per-launch DRAM bytes of a kernel on the config-2 workload from the committed
    ncu summary profiles/<name>_c2_dram_traffic.txt, valid only while the kernel's
    sources are unchanged since the capture."""
    fp = os.path.join(ROOT, "profiles", "%s_c2_dram_traffic.txt" % name)
    if not os.path.exists(fp):
        return None
    vals = {}
    for line in open(fp):
        if "=" in line and not line.startswith("#"):
            k, _, v = line.partition("=")
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash(name):
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    fp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(fp):
        try:
            return json.load(open(fp)), "measured"
        except ValueError:
            pass
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        inside = [r for r in rows if t_start - 0.06 <= r[0] <= t_end + 0.06]
        window = "timed"
        if not inside and rows:
            mid = 0.5 * (t_start + t_end)
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
            window = "nearest"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for nm, val in zip(names, r[3][5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median([r[1] for r in inside])),
                "sm_max_mhz": float(max(r[2] for r in inside)), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------- distributed


def shard_requests(B: int, world: int, rank: int):
    """Contiguous request range [lo, hi) of `rank` when one batch is split across
    ranks (requests are independent: no collective is needed on the data path)."""
    base, extra = divmod(B, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle arm


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step(batch, units, threads, packed):
    """One bounded sample of the workload on the CPU oracle: verify of the listed
    (request, head) units, the greedy walk of every request, commit of the units."""
    import oracle
    oracle.verify(batch, units=units, threads=threads, packed=packed)
    ln, path, _ = oracle.accept_batch(batch)
    oracle.commit(batch, ln, path, units=units, threads=threads, packed=packed)


def time_oracle(batch, total_steps: int, budget_s: float, threads: int, fill_budget=False):
    """Pick a sample size (units per step) so total_steps steps take about budget_s
    (fill_budget: then run as many steps of that size as fill budget_s); returns
    (node_heads_per_s, units_per_step, steps_run, seconds, threads_used)."""
    import oracle
    packed = oracle._Packed(batch)
    n_units = batch.B * batch.H
    sizes = np.diff(batch.node_offsets)
    probe = np.arange(min(n_units, max(threads * 2, 8)), dtype=np.int32)
    t0 = time.perf_counter()
    oracle_step(batch, probe, threads, packed)
    per_unit = (time.perf_counter() - t0) / len(probe)
    want = budget_s / max(total_steps, 1) / max(per_unit, 1e-9)
    upl = int(min(n_units, max(1, want)))
    units_all = np.arange(n_units, dtype=np.int32)
    if fill_budget:
        # one calibration step at that size, then as many steps as fill the budget
        t0 = time.perf_counter()
        oracle_step(batch, units_all[:upl], threads, packed)
        step_t = time.perf_counter() - t0
        total_steps = int(min(5000, max(3, budget_s / max(step_t, 1e-9))))
    t0 = time.perf_counter()
    nh = 0
    for s in range(total_steps):
        start = (s * upl) % n_units
        units = np.take(units_all, np.arange(start, start + upl), mode="wrap")
        oracle_step(batch, units, threads, packed)
        nh += int(sum(sizes[u // batch.H] for u in units))
    dt = time.perf_counter() - t0
    used = min(threads, upl)
    return nh / dt, upl, total_steps, dt, used


def run_reference(args, world, rank):
    if rank != 0:
        return
    import workloads
    b = workloads.make_config(args.config)
    threads = cpu_cores()
    steps = args.steps + args.warmup
    value, upl, n, dt, threads = time_oracle(b, steps, 60.0, threads)
    ms = dt / n * 1e3
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOADS[args.config], "B": b.B, "H": b.H, "dk": b.dk,
                       "dv": b.dv, "max_nodes": b.max_nodes},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d steps, each the fp64 oracle on %d of the %d "
                                       "(request, head) units (verify + greedy walk of all "
                                       "requests + commit)" % (n, upl, b.B * b.H)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm


ATTN_H, ATTN_HKV, ATTN_D = 32, 8, 128


def attention_setup(base, ctx, dev, stream):
    """The attention layers' share of the verification pass on `base`'s trees: 32 query
    heads over 8 KV heads, d = 128, a `ctx`-position shared prefix per request (bf16
    cache, seeded N(0, 1) values).  Returns (tree_call, decode_call, bytes_tree,
    bytes_decode, flops_tree, status); decode_call runs the same cache with one query
    node per request (the first node of its tree), as a plain decoding step would."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads
    B, T, H, Hkv, d = base.B, base.T, ATTN_H, ATTN_HKV, ATTN_D
    ai = workloads.attention_inputs(base, H, Hkv, d, [ctx] * B, P=ctx, seed=51, widen=False)
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    kc, vc = cu(ai["k_cache"]), cu(ai["v_cache"])
    del ai["k_cache"], ai["v_cache"]
    q, kt, vt, cl = cu(ai["q"]), cu(ai["k_tree"]), cu(ai["v_tree"]), cu(ai["ctx_len"])
    offs, par = cu(base.node_offsets), cu(base.parent)
    first = base.node_offsets[:-1].astype(np.int64)
    q1, kt1, vt1 = cu(ai["q"][first]), cu(ai["k_tree"][first]), cu(ai["v_tree"][first])
    offs1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    par1 = torch.full((B,), -1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((T, H, d), dtype=torch.float32, device=dev)
    out1 = torch.empty((B, H, d), dtype=torch.float32, device=dev)

    def make(Tn, maxn, o, p, qq, ktt, vtt, oo):
        wsb = tv.tv_tree_attention_workspace_bytes(B, Tn, maxn, H, Hkv, d, ctx)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device=dev) if wsb else None

        def call():
            tv.tv_tree_attention(B, Tn, maxn, H, Hkv, d, ctx, o, p, cl, qq, kc, vc, ktt, vtt,
                                 ai["scale"], oo, ws, wsb, status, stream)
        return call

    tree_call = make(T, base.max_nodes, offs, par, q, kt, vt, out)
    dec_call = make(B, 1, offs1, par1, q1, kt1, vt1, out1)
    cache = 2 * B * Hkv * ctx * d * 2
    side = lambda Tn: Tn * H * d * 2 + 2 * Tn * Hkv * d * 2 + Tn * H * d * 4 + 8 * Tn + 8 * B
    # scores and weighted values over every visible key of every query row
    path = int(np.asarray(base.depth, dtype=np.int64).sum())
    flops = 4 * H * d * (T * ctx + path)
    return tree_call, dec_call, cache + side(T), cache + side(B), flops, status


# Distributions of the per-node factors (as in the workloads module): q, k, v ~
# N(0, 1/dk), g per the configuration, H0 ~ N(0, h0 std).  The per-configuration
# block draws them on the device with a seeded torch generator, so that the 4.8 GB
# large-tree stack needs no host-side generation; the trees and token arrays come
# from the workloads module unchanged (values=False).
G_KIND = {1: "softplus01", 2: "softplus_m1", 3: "logsig16", 4: "softplus_m1", 5: "logsig16"}
H0_STD = {1: 0.1, 2: 0.05, 3: 0.05, 4: 0.05, 5: 0.05}
# ncu figures of each configuration's verify kernel (profiles/verify_configs_ncu.txt),
# valid while the kernel's sources hash to the recorded value
CONFIG_KERNEL_SOURCES = {
    3: [_CS + f for f in ("verify_tc_fdiag.cu", "tc_common.cuh", "tc_ptx.cuh", "tv_internal.cuh")],
    4: [_CS + f for f in ("verify_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "tv_internal.cuh")],
    5: [_CS + f for f in ("verify_tc_fwalk.cu", "tc_common.cuh", "tc_ptx.cuh", "tv_internal.cuh")],
}


def sources_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        fp = os.path.join(ROOT, p)
        if os.path.exists(fp):
            h.update(open(fp, "rb").read())
    return h.hexdigest()[:16]


def recorded_config_profile(cfg: int):
    """Tensor-pipe share and DRAM bytes of config cfg's verify kernel from the
    committed ncu summary, or None when absent or the sources changed."""
    fp = os.path.join(ROOT, "profiles", "verify_configs_ncu.txt")
    if cfg not in CONFIG_KERNEL_SOURCES or not os.path.exists(fp):
        return None
    for line in open(fp):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if len(f) >= 5 and f[0] == "c%d" % cfg:
            if f[1] != sources_hash(CONFIG_KERNEL_SOURCES[cfg]):
                return None
            return {"tensor_pipe_pct": float(f[2]), "dram_bytes_per_unit": float(f[3]),
                    "captured_on": f[4]}
    return None


def fill_factors(d, cfg: int, seed: int, dev):
    """Draw q, k, v, g, H0 of a DeviceBatch on the device (see G_KIND, H0_STD)."""
    import torch
    import torch.nn.functional as F
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T, H, dk, dv, B = max(d.T, 1), d.H, d.dk, d.dv, d.B
    dt = torch.bfloat16 if d.qkv_dtype == 0 else torch.float32
    sc = 1.0 / np.sqrt(dk)
    d.q = (torch.randn((T, H, dk), generator=gen, device=dev) * sc).to(dt)
    d.k = (torch.randn((T, H, dk), generator=gen, device=dev) * sc).to(dt)
    d.v = (torch.randn((T, H, dv), generator=gen, device=dev) * sc).to(dt)
    kind = G_KIND[cfg]
    if kind == "softplus01":
        d.g = -F.softplus(torch.randn((T, H), generator=gen, device=dev))
    elif kind == "softplus_m1":
        d.g = -F.softplus(torch.randn((T, H), generator=gen, device=dev) * 0.5 - 1.0)
    else:
        d.g = F.logsigmoid(torch.randn((T, H, dk), generator=gen, device=dev) + 2.0) / 16.0
    d.H0 = torch.randn((B, H, dk, dv), generator=gen, device=dev) * H0_STD[cfg]


def per_config_block(tv, dev, stream, l2, peak, skip, cfg2_us=None):
    """tv_verify at every configuration's full size: kernel, algorithmic bytes, launch
    time (graph replays over input sets rotated past 4x L2), GB/s, fraction of the
    measured HBM peak, node-heads/s, transient bytes against per-node states, and the
    tensor-pipe share of the committed ncu capture for configurations 3-5."""
    import torch
    import workloads
    out = {}
    launches = {1: 400, 2: 400, 3: 100, 4: 20, 5: 5}
    for cfg in range(1, 6):
        if cfg in skip:
            continue
        hb = workloads.make_config(cfg, seed=1000 + cfg, values=False)
        vb = verify_bytes(hb)
        R = 1 if vb >= 4 * l2 else max(2, int(np.ceil(4.0 * l2 / vb)) + 1)
        if vb < 1 << 20:
            R = 1  # a few KB: latency only
        dbs = []
        for r in range(R):
            d = tv.DeviceBatch(hb, device=dev)
            fill_factors(d, cfg, 5000 + 17 * cfg + r, dev)
            dbs.append(d)
        variant = dbs[0].variant()
        K = launches[cfg]
        with torch.cuda.stream(stream):
            for d in dbs:
                d.status.zero_()
                d.verify(stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                dbs[i % R].verify(stream=stream)
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        for d in dbs:
            if int(d.status[0].item()) != 0:
                raise SystemExit("device status %d in config %d" % (int(d.status[0].item()), cfg))
        t = e0.elapsed_time(e1) * 1e-3 / K
        qk = 2 if hb.qkv_dtype == "bf16" else 4
        sg = 4 if hb.decay == "scalar" else 4 * hb.dk
        # the token-level factors that replace per-node states: g, k and v
        factors = hb.T * hb.H * ((hb.dk + hb.dv) * qk + sg)
        naive = hb.T * hb.H * hb.dk * hb.dv * 4
        entry = {"workload": WORKLOADS[cfg], "kernel": KERNEL_NAMES.get(variant, str(variant)),
                 "bytes_per_launch": int(vb), "launch_us": t * 1e6, "gbs": vb / t / 1e9,
                 "frac": vb / t / 1e9 / peak, "node_heads_per_s": hb.T * hb.H / t,
                 "node_heads": hb.T * hb.H, "launches": K, "input_sets": R,
                 "transient_bytes": {"library_workspace": 0, "factors": int(factors),
                                     "naive_per_node_states": int(naive),
                                     "cut_vs_naive": 1.0 - factors / naive}}
        prof = recorded_config_profile(cfg)
        if prof is not None:
            entry["ncu"] = prof
        out["c%d" % cfg] = entry
        del g, dbs
        torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    tv.build()
    tv.load()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20

    cfg = args.config
    base = workloads.make_config(cfg, seed=1000 + cfg + 7919 * rank)
    per_set = verify_bytes(base) + base.B * base.H * base.dk * base.dv * 4 * 2
    # enough distinct sets that one cycle touches > 4x L2 (one set when it alone does)
    R = args.sets or (1 if per_set >= 4 * l2 else max(4, int(np.ceil(4.0 * l2 / per_set)) + 1))
    sets = [base] + [workloads.make_config(cfg, seed=1000 + cfg + 7919 * rank + 101 * r)
                     for r in range(1, R)]
    dbs = [tv.DeviceBatch(s, device=dev) for s in sets]
    stream = torch.cuda.Stream(device=dev)
    node_heads = base.T * base.H

    # target logits for the argmax + walk call (config 2's 32000-token vocabulary; the
    # others draw their tokens from 32), rows planted so the argmax is the target
    vocab = 32000 if cfg == 2 else 64
    logits = []
    for r, hb in enumerate(sets):
        rl, nl = workloads.target_logits(hb, vocab, seed=31 + r)
        logits.append((torch.from_numpy(rl.view(np.int16)).to(dev),
                       torch.from_numpy(nl.view(np.int16)).to(dev)))
    root_am = torch.empty(base.B, dtype=torch.int32, device=dev)
    tgt_am = torch.empty(max(base.T, 1), dtype=torch.int32, device=dev)

    # workspace of the naive serial baseline (per-node states), when it is modest
    serial_bytes = tv.tv_verify_serial_workspace_bytes(dbs[0].problem())
    serial_ws = (torch.empty(serial_bytes // 4, dtype=torch.float32, device=dev)
                 if 0 < serial_bytes <= 4 * 2 ** 30 else None)

    def accept_logits(i):
        d, (rl, nl) = dbs[i], logits[i]
        tv.tv_accept_greedy_logits(d.B, d.T, d.max_nodes, d.max_depth, vocab, d.node_offsets,
                                   d.parent, d.draft, rl, nl, root_am, tgt_am, d.accept_len,
                                   d.path, d.bonus, d.status, stream)

    mode = args.pipeline
    fused = mode in ("one", "fused")  # the state stays resident and is updated in place

    def step_one(d):
        # one pass of the hot path in one launch: the greedy walk of the previous tree
        # (this set's own, in the rotation), the commit of the paths it finds to the
        # resident state, and the verification of this set's tree
        d.accept_commit_verify(d, stream=stream)

    def step_fused(d):
        # one pass of the hot path: the commit of this set's previous accepted paths
        # and the verification in one launch, then the greedy walk (its paths are the
        # commit pending for the set's next step; the state stays resident in d.H0)
        d.commit_verify(d, stream=stream)
        d.accept(stream=stream)

    def step_separate(d):
        # one pass of the hot path: verify, then greedy accept + commit in one launch
        d.verify(stream=stream, variant=args.variant)
        d.accept_commit(stream=stream)

    step = {"one": step_one, "fused": step_fused, "separate": step_separate}[mode]

    with torch.cuda.stream(stream):
        for d in dbs:
            d.status.zero_()
            d.accept(stream=stream)  # the first pending commit of every set
        for w in range(args.warmup):
            step(dbs[w % R])
    stream.synchronize()
    for d, s in zip(dbs, sets):
        st = int(d.status[0].item())
        if st != 0:
            raise SystemExit("device status %d (%s) during warm-up" % (st, tv.status_string(st)))

    def capture(fn_list):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for fn in fn_list:
                fn()
        return g

    def graphs_for(kind, K):
        """Graphs whose replays launch exactly K units of `kind` cycling through the sets."""
        def one(i):
            d = dbs[i % R]
            if kind == "step":
                return lambda d=d: step(d)
            if kind == "step_separate":
                return lambda d=d: step_separate(d)
            if kind == "step_fused":
                return lambda d=d: step_fused(d)
            if kind == "step_one":
                return lambda d=d: step_one(d)
            if kind == "commit_verify":
                return lambda d=d: d.commit_verify(d, stream=stream)
            if kind == "verify":
                return lambda d=d: d.verify(stream=stream, variant=args.variant)
            if kind == "accept":
                return lambda d=d: d.accept(stream=stream)
            if kind == "serial":
                return lambda d=d: d.verify_serial(serial_ws, stream=stream)
            if kind == "accept_logits":
                return lambda i=i: accept_logits(i % R)
            if kind == "step_logits":
                return lambda d=d, i=i: (d.commit_verify(d, stream=stream), accept_logits(i % R))
            if kind == "accept_commit":
                return lambda d=d: d.accept_commit(stream=stream)
            return lambda d=d: d.commit(stream=stream)
        full = capture([one(i) for i in range(R)])
        rem = K % R
        remg = capture([one(i) for i in range(rem)]) if rem else None
        return full, K // R, remg

    def timed(kind, K):
        """Seconds for exactly K launches of `kind`, replayed on `stream` between CUDA
        events recorded on that same stream (barrier and synchronize on both sides)."""
        full, reps, remg = graphs_for(kind, K)
        with torch.cuda.stream(stream):
            full.replay()  # upload / warm
            if remg is not None:
                remg.replay()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_host0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                full.replay()
            if remg is not None:
                remg.replay()
            e1.record(stream)
        e1.synchronize()
        t_host1 = time.time()
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) * 1e-3, t_host0, t_host1

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    t_step, th0, th1 = timed("step", K)
    clocks = sampler.summary(th0, th1)
    t_verify, _, _ = timed("verify", K)
    t_accept, _, _ = timed("accept", K)
    t_commit, _, _ = timed("commit", K)
    t_acom, _, _ = timed("accept_commit", K)
    t_cv, _, _ = timed("commit_verify", K)
    t_al, _, _ = timed("accept_logits", K)
    t_ser = timed("serial", max(1, K // 8))[0] * 8 if serial_ws is not None else None
    t_sl, _, _ = timed("step_logits", K)
    t_modes = {mode: t_step}
    for m in ("one", "fused", "separate"):
        if m not in t_modes:
            t_modes[m] = timed("step_" + m, K)[0]
    t_sep = t_modes["separate"]
    sampler.stop()
    for d in dbs:
        st = int(d.status[0].item())
        if st != 0:
            raise SystemExit("device status %d (%s)" % (st, tv.status_string(st)))

    t_step_max = max_over_ranks(t_step, world)
    total_nh = sum_over_ranks(node_heads * K, world)
    value = total_nh / t_step_max
    ms_per_step = t_step_max / K * 1e3

    # ---------------- end to end through the binding with pinned host buffers
    e2e = run_e2e(args, sets[0], dev, stream, tv, world, mode)
    if mode in ("one", "fused"):
        # the same with the layer's outputs read back every step as well
        wo = run_e2e(args, sets[0], dev, stream, tv, world, mode, read_outputs=True)
        e2e["with_outputs_read_back"] = {k: wo[k] for k in ("value", "unit", "h2d_bytes_per_step",
                                                             "d2h_bytes_per_step", "ms_per_step")}

    # ---------------- one verify launch over `fold` layers folded into the head axis
    folded = {}
    if cfg == 2 and args.fold > 1 and rank == 0:
        fb = workloads.config2(seed=77, H=base.H * args.fold)
        fd = tv.DeviceBatch(fb, device=dev)
        del fb
        fb_bytes = verify_bytes_of(fd)
        auto_variant = fd.variant()
        for name, var in (("auto", args.variant), ("one_unit_kernel", 2)):
            with torch.cuda.stream(stream):
                fd.status.zero_()
                for _ in range(3):
                    fd.verify(stream=stream, variant=var)
            stream.synchronize()
            KF = max(10, min(200, K // 100))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(KF):
                    fd.verify(stream=stream, variant=var)
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            e1.synchronize()
            if int(fd.status[0].item()) != 0:
                raise SystemExit("device status %d in folded run" % int(fd.status[0].item()))
            t_f = e0.elapsed_time(e1) * 1e-3 / KF
            used = var if var else auto_variant
            folded[name] = {"layers": args.fold, "H": fd.H, "launches": KF,
                            "kernel": KERNEL_NAMES.get(used, str(used)),
                            "bytes_per_launch": fb_bytes, "launch_us": t_f * 1e6,
                            "node_heads_per_s": fd.T * fd.H / t_f,
                            "gbs": fb_bytes / t_f / 1e9}
            del g
        del fd
        torch.cuda.empty_cache()

    # ---------------- best-first draft trees (the GLA-like layer's and the large-tree
    # stack's tree shapes), one launch per batch of requests
    builder = None
    if rank == 0:
        builder = {}
        for name, (Bt, Ct, cap, nt, alpha) in (("64-node trees, B=32, depth <= 8", (32, 8, 8, 64, 0.3)),
                                               ("256-node trees, B=8, depth <= 16", (8, 8, 16, 256, 0.2))):
            marg = torch.from_numpy(np.random.default_rng(3).dirichlet(
                alpha * np.ones(Ct), size=(Bt, cap))).to(dev)
            par = torch.empty((Bt, nt), dtype=torch.int32, device=dev)
            tok = torch.empty((Bt, nt), dtype=torch.int32, device=dev)
            rho = torch.empty((Bt, nt), dtype=torch.float64, device=dev)
            cnt = torch.empty(Bt, dtype=torch.int32, device=dev)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    tv.tv_build_tree(Bt, Ct, cap, nt, marg, None, par, tok, rho, cnt, stream)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(20):
                    tv.tv_build_tree(Bt, Ct, cap, nt, marg, None, par, tok, rho, cnt, stream)
                e1.record(stream)
            e1.synchronize()
            builder[name] = {"call": "tv_build_tree", "launch_us": e0.elapsed_time(e1) * 1e3 / 20,
                             "candidates": Ct}

    # ---------------- stochastic acceptance on this workload's trees: fp32 target and
    # draft rows over `vocab` tokens, drafts drawn from the draft rows
    stochastic = None
    if rank == 0:
        sin = workloads.stochastic_inputs(base, vocab, seed=41)
        cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        sp = {k: cu(v) for k, v in sin.items()}
        sd = tv.DeviceBatch(base, device=dev)
        slen = torch.empty(base.B, dtype=torch.int32, device=dev)
        spath = torch.empty((base.B, base.max_depth), dtype=torch.int32, device=dev)
        sbon = torch.empty(base.B, dtype=torch.int32, device=dev)

        def stoch():
            tv.tv_accept_stochastic(base.B, base.T, base.max_nodes, base.max_depth, vocab,
                                    sd.node_offsets, sd.parent, sp["draft"], sp["root_p"],
                                    sp["node_p"], sp["root_q"], sp["node_q"], sp["u_accept"],
                                    sp["u_bonus"], slen, spath, sbon, sd.status, stream)
        with torch.cuda.stream(stream):
            sd.status.zero_()
            for _ in range(3):
                stoch()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(20):
                stoch()
            e1.record(stream)
        e1.synchronize()
        if int(sd.status[0].item()) != 0:
            raise SystemExit("device status %d in stochastic acceptance" % int(sd.status[0].item()))
        stochastic = {"call": "tv_accept_stochastic", "vocab": vocab,
                      "launch_us": e0.elapsed_time(e1) * 1e3 / 20,
                      "mean_accept_len": float(slen.float().mean().item()),
                      "rows_fp32_mb": (base.B + base.T) * vocab * 8 / 1e6}
        del sp, sd

    # ---------------- tree-masked softmax attention (the hybrid target's attention
    # layers) on this workload's trees, and the same cache with one query per request
    attention = None
    if rank == 0 and args.attention_ctx > 0:
        tcall, dcall, ab, db, aflops, ast = attention_setup(base, args.attention_ctx, dev, stream)

        def time_calls(call, KA=20):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    call()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(KA):
                    call()
            with torch.cuda.stream(stream):
                g.replay()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) * 1e-3 / KA

        t_at = time_calls(tcall)
        t_dec = time_calls(dcall)
        if int(ast[0].item()) != 0:
            raise SystemExit("device status %d in tree attention" % int(ast[0].item()))
        hbm = float(measured_peaks()[0].get("hbm_gbs", 6800.0))
        attention = {
            "call": "tv_tree_attention",
            "workload": "%d requests x config-2 trees (%d nodes), %d query heads over %d KV "
                        "heads, d=%d, %d-position shared prefix, bf16" % (
                            base.B, base.T, ATTN_H, ATTN_HKV, ATTN_D, args.attention_ctx),
            "launch_us": t_at * 1e6, "bytes_per_launch": ab, "gbs": ab / t_at / 1e9,
            "roofline": {"bound": "hbm", "achieved": ab / t_at / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": ab / t_at / 1e9 / hbm,
                         "traffic": recorded_traffic("tree_attention")},
            "tensor_tflops": aflops / t_at / 1e12,
            "decode_us": t_dec * 1e6, "decode_gbs": db / t_dec / 1e9,
            "tree_over_decode": t_at / t_dec,
            "l2": "the %d MB cache is over twice the L2; launches replay back to back"
                  % (ab // 2 ** 20)}
        del tcall, dcall
        torch.cuda.empty_cache()

    # ---------------- roofline of the dominant kernel of the step
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    vb = verify_bytes(base)
    v_launch = t_verify / K
    lens = [int(x) for x in dbs[0].accept_len[:base.B].cpu().numpy()]
    cb = commit_bytes(base, lens)
    cvb = commit_verify_bytes(base, lens)
    # logits rows read once, tree arrays, acceptance outputs and argmax outputs
    al_bytes = ((base.B + base.T) * vocab * 2 + 8 * base.T + 4 * (base.B + 1)
                + 4 * base.B * (3 + base.max_depth) + 4 * base.T)
    cv_launch = t_cv / K
    used_variant = args.variant if args.variant else dbs[0].variant()
    # the recorded captures are of the fused tensor-core kernel on the config-2 workload
    tc2 = cfg == 2 and used_variant == 3
    if mode == "one":
        # the step is the one launch
        dom_bytes, dom_t = accept_commit_verify_bytes(base, lens), t_step / K
        dom_name = "tv_accept_commit_verify"
        traffic = recorded_traffic("accept_commit_verify") if tc2 else None
    elif fused:
        dom_bytes, dom_t, dom_name = cvb, cv_launch, "tv_commit_verify"
        traffic = recorded_traffic("commit_verify") if tc2 else None
    else:
        dom_bytes, dom_t, dom_name = vb, v_launch, "tv_verify"
        traffic = recorded_traffic("verify") if tc2 else None
    achieved = dom_bytes / dom_t / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": dom_name, "bytes_per_launch": dom_bytes,
                "launch_us": dom_t * 1e6, "peak_kind": "%s (hbm_gbs burst copy)" % peak_kind}

    # context for the roofline: a plain torch read reduction (torch.sum) over the same
    # number of bytes, timed the same way (graph replays, regions rotated past 4x L2);
    # at a few tens of MB one launch of any streaming kernel is dominated by launch and
    # first-byte latency, so this is the practical ceiling at the step's size
    same_bytes = None
    if rank == 0:
        nfl = max(1, int(dom_bytes) // 4)
        R2 = 1 if dom_bytes >= 4 * l2 else max(4, int(4 * l2 / max(dom_bytes, 1)) + 1)
        pool = torch.ones(R2 * nfl, dtype=torch.float32, device=dev)
        acc = torch.empty((), dtype=torch.float32, device=dev)
        KS2 = R2 * max(1, 200 // R2)
        with torch.cuda.stream(stream):
            torch.sum(pool[:nfl], dim=0, out=acc)
        stream.synchronize()
        gs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gs, stream=stream):
            for k in range(KS2):
                torch.sum(pool[(k % R2) * nfl:(k % R2 + 1) * nfl], dim=0, out=acc)
        with torch.cuda.stream(stream):
            gs.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gs.replay()
            e1.record(stream)
        e1.synchronize()
        t_sum = e0.elapsed_time(e1) * 1e-3 / KS2
        same_bytes = {"what": "torch.sum over the dominant kernel's byte count", "bytes": int(dom_bytes),
                      "launch_us": t_sum * 1e6, "gbs": dom_bytes / t_sum / 1e9,
                      "frac": dom_bytes / t_sum / 1e9 / peak,
                      "ours_over_it": t_sum / dom_t}
        del gs, pool
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_cores()
        v, upl, n, dt, threads = time_oracle(base, 40, 15.0, threads, fill_budget=True)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d steps of the fp64 oracle, each on %d of the %d (request, head) "
                         "units (verify + greedy walk + commit), %.1f s" % (n, upl,
                                                                              base.B * base.H,
                                                                              dt)}
        v1, upl1, n1, dt1, _ = time_oracle(base, 20, 5.0, 1, fill_budget=True)
        cpu["one_thread"] = {"value": v1, "unit": UNIT, "cores": 1,
                             "sample": "%d steps, each on %d units, %.1f s" % (n1, upl1, dt1)}

    # host time of one un-captured call (argument checks, tensor maps, launch)
    host_call = None
    configs = None
    if rank == 0:
        host_call = {}
        for name, fn in (("tv_verify", lambda: dbs[0].verify(stream=stream)),
                         ("tv_commit_verify", lambda: dbs[0].commit_verify(dbs[0], stream=stream)),
                         ("tv_accept_commit_verify",
                          lambda: dbs[0].accept_commit_verify(dbs[0], stream=stream))):
            for _ in range(20):
                fn()
            stream.synchronize()
            NC = 300
            t0 = time.perf_counter()
            for _ in range(NC):
                fn()
            t1 = time.perf_counter()
            stream.synchronize()
            host_call[name] = (t1 - t0) / NC * 1e6
        host_call["unit"] = "us of host time per call, not captured in a graph"
        if not args.no_configs:
            configs = per_config_block(tv, dev, stream, l2, peak, skip=set())

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOADS[cfg], "B": base.B, "H": base.H, "dk": base.dk,
                       "dv": base.dv, "max_nodes": base.max_nodes,
                       "node_heads_per_step": node_heads,
                       "verify_kernel": KERNEL_NAMES.get(used_variant, str(used_variant)),
                       "pipeline": {"one": "tv_accept_commit_verify (one launch: the previous "
                                           "tree's greedy walk, its commit, this tree's "
                                           "verification); state resident in HBM, updated "
                                           "in place",
                                    "fused": "tv_commit_verify + tv_accept_greedy; state "
                                             "resident in HBM, updated in place",
                                    "separate": "tv_verify + tv_accept_commit"}[mode],
                       "inputs": "bf16 q/k/v, fp32 g/H0/out/H_new",
                       "l2": "inputs larger than L2: %d input sets rotated, %.0f MB touched per "
                             "cycle vs %.0f MB L2" % (R, R * per_set / 1e6, l2 / 1e6),
                       "timing": "CUDA graph replays of the K steps, CUDA events on the "
                                 "launching stream"},
            "roofline": roofline,
            "same_bytes_read_reduction": same_bytes,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (1 if mode == "one" else 2) * K,
            "clocks": clocks,
            "kernels_us": {"verify": t_verify / K * 1e6, "accept_commit": t_acom / K * 1e6,
                           "commit_verify": t_cv / K * 1e6,
                           "accept (separate call)": t_accept / K * 1e6,
                           "commit (separate call)": t_commit / K * 1e6},
            "step_kernels": {"one": ["tv_accept_commit_verify"],
                             "fused": ["tv_commit_verify", "tv_accept_greedy"],
                             "separate": ["tv_verify", "tv_accept_commit"]}[mode],
            "step_us": {m: t / K * 1e6 for m, t in t_modes.items()},
            "verify_only": {"value": node_heads / v_launch, "unit": UNIT,
                            "gbs": vb / v_launch / 1e9, "bytes_per_launch": vb,
                            "frac": vb / v_launch / 1e9 / peak,
                            "traffic": recorded_traffic("verify") if tc2 else None},
            "verify_folded_layers": ({k: dict(v, frac=v["gbs"] / peak)
                                      for k, v in folded.items()} if folded else None),
            "commit_gbs": cb / (t_commit / K) / 1e9,
            "speedup_over_serial": ({
                "serial_us": t_ser / K * 1e6, "tree_closed_form_us": t_verify / K * 1e6,
                "ratio": t_ser / t_verify,
                "serial": "tv_verify_serial: node after node, per-node states in a %d MB "
                          "workspace" % (serial_bytes // 2 ** 20)}
                if t_ser is not None else None),
            "host_us_per_call": host_call,
            "per_config": configs,
            "tree_builder": builder,
            "stochastic_accept": stochastic,
            "tree_attention": attention,
            "accept_from_logits": {
                "call": "tv_accept_greedy_logits", "vocab": vocab,
                "bytes_per_launch": al_bytes, "launch_us": t_al / K * 1e6,
                "gbs": al_bytes / (t_al / K) / 1e9,
                "frac": al_bytes / (t_al / K) / 1e9 / peak,
                "step_us_with_it": t_sl / K * 1e6,
                "step": "tv_commit_verify + tv_accept_greedy_logits"},
            "transient_bytes": {"library_workspace": 0,
                                # the token-level factors g, k, v kept instead of states
                                "factors": int(base.T * base.H * (
                                    (base.dk + base.dv) * (2 if base.qkv_dtype == "bf16" else 4)
                                    + (4 if base.decay == "scalar" else 4 * base.dk))),
                                "naive_per_node_states": int(base.T * base.H * base.dk * base.dv
                                                             * 4)},
        }
        print(json.dumps(line), flush=True)


def run_e2e(args, host_batch, dev, stream, tv, world, mode, read_outputs=False):
    """The step through the binding with host buffers: pinned host -> device copies
    of the step's inputs, the calls, device -> pinned host copies of its results.
    One-launch and fused pipelines: the state is resident on the device (the commit
    updates it in place), so the inputs are the tree, factors and tokens, and the
    results the host needs are the acceptance (lengths, paths, bonus tokens) and the
    status; the layer's outputs stay in HBM for the next layer unless `read_outputs`
    asks for them too.  Separate pipeline: the state is copied in and H_new and the
    outputs out.  In the one-launch pipeline a step's acceptance results are the walk
    of the previous step's tree, written to the step's own result buffers.

    Each step moves one contiguous staging range in and one out.  Four staging sets
    rotate over four streams, as a decode loop would run them: set s % 4 was last read
    by the kernels of step s - 3 (as their pending commit), so the input copy of step s
    waits only for those and overlaps the kernels of steps s - 2 and s - 1; the kernels
    of a step wait for those of the previous step (the state and the pending commit
    chain through them)."""
    import torch
    fused = mode in ("one", "fused")
    ins = ["node_offsets", "parent", "depth", "q", "k", "v", "g", "draft", "target",
           "root_argmax"]
    outs = ["out", "accept_len", "path", "bonus"]
    if not fused:
        ins.append("H0")
        outs.append("H_new")
    elif not read_outputs:
        outs = ["accept_len", "path", "bonus"]
    # one staging layout on both sides: the step's inputs, the status word and the
    # results (then the outputs, where they are not read back); the batch's tensors
    # become views into it.  The status travels both ways, so an error in any step
    # stays set and is caught after the timed region.
    names = ins + ["status"] + outs + ([] if "out" in outs else ["out"])
    probe = tv.DeviceBatch(host_batch, device=dev)
    offs, pos = {}, 0
    for n in names:
        pos = (pos + 255) // 256 * 256
        offs[n] = pos
        t = getattr(probe, n)
        pos += t.numel() * t.element_size()
    total = (pos + 255) // 256 * 256
    in_end = offs["status"] + probe.status.numel() * probe.status.element_size()
    out_begin = offs["status"]
    out_end = total if "out" in outs else offs["out"]
    del probe

    def staged():
        hb = tv.DeviceBatch(host_batch, pin=True)
        db = tv.DeviceBatch(host_batch, device=dev)
        h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
        d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
        for obj, buf in ((hb, h_stage), (db, d_stage)):
            for n in names:
                t = getattr(obj, n)
                nb = t.numel() * t.element_size()
                view = buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
                view.copy_(t if n != "status" else torch.zeros_like(t))
                setattr(obj, n, view)
        return hb, db, h_stage, d_stage

    NS = 4
    sets = [staged() for _ in range(NS)]
    if fused:
        for i in range(1, NS):
            sets[i][1].H0 = sets[0][1].H0  # one resident state
    streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(NS - 1)]
    kev = [torch.cuda.Event() for _ in range(NS)]  # kernels of the step that last used a set
    h2d = in_end
    d2h = out_end - out_begin
    # about 2 GB of host<->device traffic at most (at least 3 steps)
    K = max(NS, min(args.e2e_steps, max(3, int(2e9 / max(h2d + d2h, 1)))))

    def step(s, first=0):
        """Enqueue step s; waits on steps before `first` are left out (inside a
        captured rotation those come from the previous replay, already complete)."""
        i = s % NS
        hb, db, hs, ds = sets[i]
        st = streams[i]
        with torch.cuda.stream(st):
            if s - (NS - 1) >= first:
                st.wait_event(kev[(s - (NS - 1)) % NS])
            ds[:in_end].copy_(hs[:in_end], non_blocking=True)
            if s - 1 >= first:
                st.wait_event(kev[(s - 1) % NS])
            if mode == "one":
                db.accept_commit_verify(sets[(s - 1) % NS][1], stream=st)
            elif fused:
                db.commit_verify(sets[(s - 1) % NS][1], stream=st)
                db.accept(stream=st)
            else:
                db.verify(stream=st, variant=args.variant)
                db.accept_commit(stream=st)
            kev[i].record(st)
            hs[out_begin:out_end].copy_(ds[out_begin:out_end], non_blocking=True)

    def join_into_first():
        for st in streams[1:]:
            ev = torch.cuda.Event()
            ev.record(st)
            streams[0].wait_event(ev)

    with torch.cuda.stream(streams[NS - 1]):
        sets[NS - 1][1].accept(stream=streams[NS - 1])  # the first pending commit
    torch.cuda.synchronize()
    for s in range(2 * NS):
        step(s)
    torch.cuda.synchronize()
    # ROT rotations (NS steps each, one per set) as one CUDA graph: fork to the other
    # streams, the steps with their cross-stream waits, join back.  Replays of a graph
    # on one stream run one after the other, so the copy pipeline drains only once
    # per ROT * NS steps.
    ROT = max(1, min(33, K // NS))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=streams[0]):
        fork = torch.cuda.Event()
        fork.record(streams[0])
        for st in streams[1:]:
            st.wait_event(fork)
        for s in range(NS * ROT):
            step(s, first=0)
        join_into_first()
    with torch.cuda.stream(streams[0]):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    R = max(1, K // (NS * ROT))
    K = R * NS * ROT
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(streams[0]):
        e0.record(streams[0])
        for _ in range(R):
            g.replay()
        e1.record(streams[0])
    e1.synchronize()
    torch.cuda.synchronize()
    dt = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world)
    for hb, _, _, _ in sets:
        if int(hb.status[0]) != 0:
            raise SystemExit("device status %d in e2e" % int(hb.status[0]))
    nh = sum_over_ranks(host_batch.T * host_batch.H * K, world)
    return {"value": nh / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": K, "ms_per_step": dt / K * 1e3,
            "state": "resident in HBM" if fused else "copied in and out every step",
            "results_read": "+".join(["status"] + outs),
            "copies": "one host-to-device copy of the step's inputs and one device-to-host "
                      "copy of its results per step (one staging layout, 256-byte aligned "
                      "fields); four staging sets on four streams, so a step's input "
                      "copy overlaps the previous steps' kernels and the copies of the "
                      "other direction; %d steps replay as one CUDA graph" % (NS * ROT)}


def profile_folded(args):
    """Three verify launches over `--fold` folded config-2 layers (for ncu captures)."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads
    tv.build()
    tv.load()
    fd = tv.DeviceBatch(workloads.config2(seed=77, H=24 * args.fold))
    fd.status.zero_()
    for _ in range(3):
        fd.verify(variant=args.profile_folded)
    torch.cuda.synchronize()
    st = int(fd.status[0].item())
    print(json.dumps({"profile_folded": args.profile_folded, "layers": args.fold, "status": st}))
    if st != 0:
        raise SystemExit("device status %d" % st)


def profile_attention(args):
    """Three tree-attention launches of the attention workload (for ncu captures)."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads
    tv.build()
    tv.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    tcall, _, _, _, _, st = attention_setup(workloads.make_config(args.config, seed=1000 + args.config
                                                                  ), args.attention_ctx, dev,
                                            stream)
    for _ in range(3):
        tcall()
    torch.cuda.synchronize()
    print(json.dumps({"profile_attention": args.attention_ctx, "status": int(st[0].item())}))
    if int(st[0].item()) != 0:
        raise SystemExit("device status %d" % int(st[0].item()))


def profile_verify(args):
    """Three verify launches of one variant on the configuration's workload (for ncu)."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads
    tv.build()
    tv.load()
    if args.config == 5:
        b = workloads.config5(B=8, layers=2, heads=32)
    else:
        b = workloads.make_config(args.config)
    d = tv.DeviceBatch(b)
    d.status.zero_()
    for _ in range(3):
        d.verify(variant=args.profile_verify)
    torch.cuda.synchronize()
    st = int(d.status[0].item())
    print(json.dumps({"profile_verify": args.profile_verify, "config": args.config,
                      "units": b.B * b.H, "status": st}))
    if st != 0:
        raise SystemExit("device status %d" % st)


def profile_extras(args):
    """Three launches each of tv_build_tree (the 256-node trees, B=8) and
    tv_accept_stochastic (config-2 trees, 32000 tokens), for ncu captures."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    import workloads
    tv.build()
    tv.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    Bt, Ct, cap, nt = 8, 8, 16, 256
    marg = torch.from_numpy(np.random.default_rng(3).dirichlet(0.2 * np.ones(Ct), size=(Bt, cap))).to(dev)
    par = torch.empty((Bt, nt), dtype=torch.int32, device=dev)
    tok = torch.empty((Bt, nt), dtype=torch.int32, device=dev)
    rho = torch.empty((Bt, nt), dtype=torch.float64, device=dev)
    cnt = torch.empty(Bt, dtype=torch.int32, device=dev)
    for _ in range(3):
        tv.tv_build_tree(Bt, Ct, cap, nt, marg, None, par, tok, rho, cnt, stream)
    base = workloads.make_config(2, seed=1002)  # the trees of the default bench run
    vocab = 32000
    sin = workloads.stochastic_inputs(base, vocab, seed=41)
    sp = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in sin.items()}
    sd = tv.DeviceBatch(base, device=dev)
    sd.status.zero_()
    slen = torch.empty(base.B, dtype=torch.int32, device=dev)
    spath = torch.empty((base.B, base.max_depth), dtype=torch.int32, device=dev)
    sbon = torch.empty(base.B, dtype=torch.int32, device=dev)
    for _ in range(3):
        tv.tv_accept_stochastic(base.B, base.T, base.max_nodes, base.max_depth, vocab,
                                sd.node_offsets, sd.parent, sp["draft"], sp["root_p"], sp["node_p"],
                                sp["root_q"], sp["node_q"], sp["u_accept"], sp["u_bonus"], slen,
                                spath, sbon, sd.status, stream)
    torch.cuda.synchronize()
    st = int(sd.status[0].item())
    print(json.dumps({"profile_extras": True, "tree_counts": cnt.tolist(), "status": st}))
    if st != 0:
        raise SystemExit("device status %d" % st)


def main():
    args = parse()
    if args.profile_extras:
        profile_extras(args)
        return
    if args.profile_verify is not None:
        profile_verify(args)
        return
    if args.profile_attention:
        profile_attention(args)
        return
    if args.profile_folded is not None:
        profile_folded(args)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
