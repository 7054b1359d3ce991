"""Benchmark of the verification step on one GB300 (or N replicas).

Default workload: B=64 sequences, K=5 drafts, V=128256, bf16 logits, fused
temperature-0.8 softmax, rejection sampling (one sv_accept_from_logits call
per step).  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config config2]
    python bench.py --impl reference      # the CPU oracle on the host cores

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; between timed steps the L2 is flushed by writing a
512 MB buffer (then reading another one so no dirty lines are left), outside
the events.  SM clocks are sampled with nvidia-smi during the timed region.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIG_TEXT = {
    "config1": "B=1 K=4 V=32000 f32 probabilities, rejection sampling (600 rounds as B=600)",
    "config2": "B=64 K=5 V=128256 bf16 logits, temperature 0.8, rejection sampling",
    "config3": "B=256 K=4 V=152064 f32 probabilities, greedy",
    "config4": "B=32 ragged K_b~U{0..8} V=129280 f32 probabilities, rejection sampling",
    "config5": "B=1024 K=3 V=32000 f16 logits, half greedy / half sampled",
    "filter": "config 2 rows (B=64 K=5 V=128256 bf16 logits, T=0.8) with top-k 50 and top-p 0.9 "
              "on every sequence: one call (the fused top-k plan; floors and floored verification "
              "only for the sequences it hands on)",
    "greedy2": "B=64 K=5 V=128256 bf16 logits, greedy (each draft token the argmax of its bf16 "
               "draft row)",
    "latency1": "B=1 K=4 V=32000 f32 probabilities, rejection sampling: one B=1 call per round "
                "(the 600 rounds of config 1 in turn)",
    "long16": "B=8 K=16 V=128256 bf16 logits, temperature 0.8, draft = target + N(0, 0.3^2) (long "
              "accepted chains): the row-parallel plan",
}
WORKLOAD_OVERRIDES = {"long16": dict(B=8, K=16, draft_noise=0.3)}
FILTER_TOP_K, FILTER_TOP_P = 50, 0.9
KERNEL_NAMES = {
    "config1": "sv_verify_kernel<1, float, false>",
    "config2": "sv_verify_kernel<2, __nv_bfloat16, false>",
    "config3": "sv_verify_kernel<0, float, false>",
    "config4": "sv_verify_kernel<1, float, false>",
    "config5": "sv_verify_kernel<2, __half, false>",
    "filter": "sv_rows_kernel<2, __nv_bfloat16, true, true>",
    "greedy2": "sv_verify_kernel<0, __nv_bfloat16, false>",
    "latency1": "sv_verify_kernel<1, float, false>",
    "long16": "sv_rows_kernel<2, __nv_bfloat16, false>",
}
METRIC = "verified rows/s and achieved HBM GB/s vs GB300 peak at B=64 K=5 V=128256"
# ncu summaries that carry the dominant kernel's DRAM bytes per launch, and
# the sources that kernel and its launch plan are built from
_CSRC = os.path.join(ROOT, "speculative_decoding_verification_decode_gb300", "csrc")
PROFILE_FILES = {
    "config2": ("sv_verify_kernel_config2_traffic.md", ("sv_api.cu", "sv_kernel.cuh", "sv_verify.cuh", "sv_ptx.cuh")),
    "long16": ("sv_rows_kernel_long16_traffic.md",
               ("sv_api.cu", "sv_kernel.cuh", "sv_verify.cuh", "sv_ptx.cuh", "sv_rows.cuh", "sv_rows.cu")),
    "filter": ("sv_rows_kernel_filter_config2_traffic.md",
               ("sv_api.cu", "sv_kernel.cuh", "sv_verify.cuh", "sv_ptx.cuh", "sv_rows.cuh", "sv_rows.cu",
                "sv_topk.cuh")),
}


def kernel_source_sha(config="config2"):
    h = hashlib.sha256()
    for f in PROFILE_FILES[config][1]:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def profiled_traffic(config):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel source (else None)."""
    if config not in PROFILE_FILES:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", PROFILE_FILES[config][0])).read()
    except OSError:
        return None
    sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not sha or not val or sha.group(1) != kernel_source_sha(config):
        return None
    return int(val.group(1))


# ------------------------------------------------------------------ distributed plumbing

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist if world > 1 else None


def max_over_ranks(value, dist, device=None):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, path=None):
        """Samples `index`'s clocks every 100 ms into `path` (a temporary
        file, removed after reading, when None)."""
        self.index = index
        self.proc = None
        self.keep = path is not None
        if path is None:
            fd, path = tempfile.mkstemp(prefix=f"sv_clocks_{index}_", suffix=".csv")
            os.close(fd)
        self.path = path
        self.lines = []

    def __enter__(self):
        if os.path.dirname(self.path):
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            with open(self.path) as fh:
                self.lines = fh.readlines()
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ workload helpers

def device_inputs(wl, torch, dev):
    def td(a, dt=None):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if dt == "bf16":
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)
    x = dict(target=td(wl.target, wl.dtype), draft=td(wl.draft, wl.dtype), tokens=td(wl.tokens),
             uniforms=td(wl.uniforms), cu_k=td(wl.cu_k), temperature=td(wl.temperature),
             top_k=td(getattr(wl, "top_k", None)), top_p=td(getattr(wl, "top_p", None)))
    if x["top_k"] is not None:  # the floors' buffers, reused every step
        x["floors"] = (torch.empty(wl.target.shape[0], dtype=torch.float32, device=dev),
                       torch.empty(wl.draft.shape[0], dtype=torch.float32, device=dev))
    return x


def host_inputs(wl, torch):
    def th(a, dt=None):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
        return t.pin_memory()
    return dict(target=th(wl.target, wl.dtype), draft=th(wl.draft, wl.dtype), tokens=th(wl.tokens),
                uniforms=th(wl.uniforms), cu_k=th(wl.cu_k), temperature=th(wl.temperature),
                top_k=th(getattr(wl, "top_k", None)), top_p=th(getattr(wl, "top_p", None)))


def call(sv, wl, x):
    k = wl.K if wl.cu_k is not None else None
    if wl.mode == "greedy":
        return sv.verify_greedy(x["target"], x["tokens"], x["cu_k"], k)
    if wl.mode in ("accept", "both"):
        return sv.accept(x["target"], x["draft"], x["tokens"], x["uniforms"], x["cu_k"], k)
    if x.get("top_k") is not None:  # one call: the fused plan or the two steps, by shape
        return sv.accept_from_logits(x["target"], x["draft"], x["temperature"], x["tokens"],
                                     x["uniforms"], x["cu_k"], k, top_k=x["top_k"], top_p=x["top_p"])
    return sv.accept_from_logits(x["target"], x["draft"], x["temperature"], x["tokens"],
                                 x["uniforms"], x["cu_k"], k)


def floors(sv, wl, x):
    return sv.sampler_floors(x["target"], x["draft"], x["temperature"], x["top_k"], x["top_p"], x["cu_k"],
                             wl.K, int(wl.tokens.size), out=x["floors"])


def two_steps(sv, wl, x):
    """The filtered verification as two steps (every row's floors, then the
    floored verification), for comparison with the call's own plan."""
    k = wl.K if wl.cu_k is not None else None
    return sv.accept_from_logits(x["target"], x["draft"], x["temperature"], x["tokens"], x["uniforms"],
                                 x["cu_k"], k, top_k=x["top_k"], top_p=x["top_p"], flags=sv.FLAG_PLAN_CHAIN)


def make_workload(name, seed_shift=0):
    """A named workload; 'filter' is config 2 with top-k 50 and top-p 0.9 on
    every sequence (the sampler filters before verification)."""
    import workloads
    base = {"filter": "config2", "latency1": "config1", "long16": "config2"}.get(name, name)
    base_seed = {"config1": 1, "config2": 2, "config3": 3, "config4": 4, "config5": 5,
                 "greedy2": 6}[base]
    wl = workloads.make_config(base, seed=workloads.configs.SEED_BASE + base_seed + seed_shift,
                               **WORKLOAD_OVERRIDES.get(name, {}))
    if name == "filter":
        wl.top_k = np.full(wl.B, FILTER_TOP_K, np.int32)
        wl.top_p = np.full(wl.B, FILTER_TOP_P, np.float32)
    return wl


def algorithmic_bytes(wl, n_acc):
    """Bytes the method must move with early exit: target rows 0..n_b and
    draft rows 0..min(n_b, K_b - 1) of every sampled sequence (the resident
    row pair serves the residual / bonus scan, so nothing is read twice);
    target rows 0..n_b of greedy sequences."""
    return int(algorithmic_bytes_per_seq(wl, n_acc).sum())


def algorithmic_bytes_per_seq(wl, n_acc):
    kb = wl.k_per_seq
    n = n_acc.astype(np.int64)
    t_rows = n + 1
    if wl.mode == "greedy":
        d_rows = np.zeros_like(n)
    else:
        d_rows = np.minimum(n + 1, kb)
        if wl.temperature is not None:
            d_rows = np.where(wl.temperature > 0, d_rows, 0)
    return (t_rows + d_rows) * wl.V * wl.elem_size


def oracle_rows_per_s(wl, budget_s=20.0):
    """The CPU oracle as it stands on a bounded prefix of the batch (one core)."""
    import oracle
    kb = wl.k_per_seq
    t_start = time.perf_counter()
    done_rows = 0
    done_seq = 0
    tr0 = 0
    dr0 = 0
    while done_seq < wl.B and time.perf_counter() - t_start < budget_s:
        b = done_seq
        k = int(kb[b])
        tsl = slice(tr0, tr0 + k + 1)
        dsl = slice(dr0, dr0 + k)
        if wl.mode == "greedy":
            oracle.verify_greedy(wl.target[tsl], wl.dtype, wl.tokens[dsl], 1, k)
        elif wl.mode in ("accept", "both"):
            oracle.accept(wl.target[tsl], wl.draft[dsl], wl.tokens[dsl], wl.uniforms[tsl], 1, k)
        else:
            tk, tp = getattr(wl, "top_k", None), getattr(wl, "top_p", None)
            oracle.accept_from_logits(wl.target[tsl], wl.draft[dsl], wl.dtype,
                                      wl.temperature[b:b + 1], wl.tokens[dsl], wl.uniforms[tsl], 1, k,
                                      top_k=None if tk is None else tk[b:b + 1],
                                      top_p=None if tp is None else tp[b:b + 1])
        done_rows += k + 1
        done_seq += 1
        tr0 += k + 1
        dr0 += k
    dt = time.perf_counter() - t_start
    return done_rows / dt, done_seq, dt


# ------------------------------------------------------------------ arms

def round_view(x, wl, r):
    """Inputs of round r of a batch of independent B=1 rounds (views, no copy)."""
    K = wl.K
    out = dict(x)
    out["target"] = x["target"][r * (K + 1):(r + 1) * (K + 1)]
    out["draft"] = x["draft"][r * K:(r + 1) * K]
    out["tokens"] = x["tokens"][r * K:(r + 1) * K]
    out["uniforms"] = x["uniforms"][r * (K + 1):(r + 1) * (K + 1)]
    return out


def timed_steps(torch, stream, steps, flush, step_fn):
    """Device time of each step (CUDA events on the launching stream), the
    L2 flushed before each one."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step_fn(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def mode_summary(torch, sv, dev, stream, flush, name, steps, warmup, peak):
    """One more workload timed the same way (device time, L2 flushed between
    steps): its per-round time and bandwidth, for the main line's `modes`."""
    wl = make_workload(name)
    x = device_inputs(wl, torch, dev)
    if name == "latency1":
        n_acc = call(sv, wl, x).n_accepted.cpu().numpy()
        per_seq = algorithmic_bytes_per_seq(wl, n_acc)
        for i in range(warmup):
            call(sv, wl, round_view(x, wl, i % wl.B))
        ms = timed_steps(torch, stream, steps, flush, lambda i: call(sv, wl, round_view(x, wl, i % wl.B)))
        greedy_ms = timed_steps(torch, stream, steps, flush, lambda i: sv.verify_greedy(
            round_view(x, wl, i % wl.B)["target"], round_view(x, wl, i % wl.B)["tokens"]))
        t = float(np.mean(ms))
        alg = float(np.mean([per_seq[i % wl.B] for i in range(steps)]))
        return {"workload": CONFIG_TEXT[name], "us_per_round_sampled": t * 1e3,
                "us_per_round_greedy": float(np.mean(greedy_ms)) * 1e3,
                "rows_per_s_sampled": (wl.K + 1) / (t * 1e-3),
                "algorithmic_gbs_sampled": alg / (t * 1e-3) / 1e9,
                "rounds": f"{steps} rounds, each one B=1 call"}
    for _ in range(warmup):
        r = call(sv, wl, x)
    torch.cuda.synchronize()
    n_acc = r.n_accepted.cpu().numpy()
    t = float(np.mean(timed_steps(torch, stream, steps, flush, lambda i: call(sv, wl, x))))
    alg = algorithmic_bytes(wl, n_acc)
    formula = wl.formula_bytes()
    return {"workload": CONFIG_TEXT[name], "us_per_round": t * 1e3,
            "rows_per_s": int((wl.k_per_seq + 1).sum()) / (t * 1e-3),
            "mean_accepted": float(n_acc.mean()),
            "formula_gbs": formula / (t * 1e-3) / 1e9, "formula_frac": formula / (t * 1e-3) / 1e9 / peak,
            "algorithmic_gbs": alg / (t * 1e-3) / 1e9, "algorithmic_frac": alg / (t * 1e-3) / 1e9 / peak,
            "kernel": KERNEL_NAMES[name]}


def run_gpu(args):
    import torch

    import speculative_decoding_verification_decode_gb300 as sv
    from speculative_decoding_verification_decode_gb300._build import build

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build()
    sv.load_library()

    # every rank verifies its own batch (independent sequences: weak scaling)
    wl = make_workload(args.config, seed_shift=rank * 1000)
    x = device_inputs(wl, torch, dev)
    per_round = args.config == "latency1"  # one B=1 call per step
    step_x = (lambda i: round_view(x, wl, i % wl.B)) if per_round else (lambda i: x)
    rows_per_step = wl.K + 1 if per_round else int((wl.k_per_seq + 1).sum())
    seqs_per_step = 1 if per_round else wl.B
    stream = torch.cuda.current_stream(dev)

    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1)
        flush_r.sum()

    n_acc = call(sv, wl, x).n_accepted.cpu().numpy()  # every sequence (round) once
    for i in range(args.warmup):
        flush()
        call(sv, wl, step_x(i))
    torch.cuda.synchronize(dev)

    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local, args.clocks_csv) as clocks:
        per_step_ms = timed_steps(torch, stream, args.steps, flush, lambda i: call(sv, wl, step_x(i)))
    barrier(dist, dev)
    ms_local = float(np.mean(per_step_ms))
    ms = max_over_ranks(ms_local, dist, dev)
    floors_ms = two_ms = None
    if args.config == "filter":  # the two steps and their floors kernel, for comparison
        floors_ms = float(np.mean(timed_steps(torch, stream, args.steps, flush, lambda i: floors(sv, wl, x))))
        two_ms = float(np.mean(timed_steps(torch, stream, args.steps, flush, lambda i: two_steps(sv, wl, x))))

    # end to end through the public API with pinned host buffers
    hx = host_inputs(wl, torch)
    step_hx = (lambda i: round_view(hx, wl, i % wl.B)) if per_round else (lambda i: hx)
    h2d = sum(t.numel() * t.element_size() for t in step_hx(0).values() if t is not None)
    d2h = 3 * seqs_per_step * 4
    for i in range(2):
        call(sv, wl, step_hx(i))
    torch.cuda.synchronize(dev)
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 20))
    barrier(dist, dev)
    e_s.record(stream)
    for i in range(e2e_steps):
        rr = call(sv, wl, step_hx(i))
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, dist, dev)
    last = (e2e_steps - 1) % wl.B if per_round else None
    assert np.array_equal(rr.n_accepted.numpy(), n_acc[last:last + 1] if per_round else n_acc)

    result = None
    if rank == 0:
        peak, peak_kind = measured_peak_gbs()
        if per_round:
            per_seq = algorithmic_bytes_per_seq(wl, n_acc)
            alg = float(np.mean([per_seq[i % wl.B] for i in range(args.steps)]))
            formula = wl.formula_bytes() / wl.B
        else:
            alg = algorithmic_bytes(wl, n_acc)
            formula = wl.formula_bytes()
        achieved = alg / (ms_local * 1e-3) / 1e9
        traffic = profiled_traffic(args.config)
        value = world * rows_per_step / (ms * 1e-3)
        cpu_val, cpu_seq, cpu_dt = oracle_rows_per_s(wl, budget_s=args.cpu_budget)
        modes = None
        if args.config == "config2" and not args.no_modes:
            # the other mode at the same shape, and config 1 as single-sequence
            # rounds, each measured the same way after the main line
            modes = {name: mode_summary(torch, sv, dev, stream, flush, name, args.steps, args.warmup, peak)
                     for name in ("greedy2", "latency1", "long16")}
        result = {
            "metric": METRIC,
            "value": value,
            "unit": "verified rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded Philox; shapes and distributions of the workload)",
            "config": {
                "workload": f"{args.config}: {CONFIG_TEXT[args.config]}",
                "B": 1 if per_round else wl.B, "K": wl.K, "V": wl.V, "input_dtype": wl.dtype,
                "rows_per_step": rows_per_step,
                "rounds_per_s": world * seqs_per_step / (ms * 1e-3),
                "us_per_round": ms * 1e3 / seqs_per_step,
                "mean_accepted": float(n_acc.mean()),
                "formula_bytes_per_step": formula,
                "formula_gbs": formula / (ms * 1e-3) / 1e9,
                "algorithmic_bytes_per_step": alg,
                "l2": "flushed between timed steps (512 MB write, then a 512 MB read)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                **({"two_steps_us": two_ms * 1e3, "two_steps_floors_us": floors_ms * 1e3,
                    "two_steps_floors_gbs": formula / (floors_ms * 1e-3) / 1e9,
                    "top_k": FILTER_TOP_K, "top_p": FILTER_TOP_P} if floors_ms is not None else {}),
            },
            "roofline": {
                "bound": "hbm",
                "kernel": KERNEL_NAMES[args.config],
                "achieved": achieved,
                "peak": peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst)",
                "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": traffic,
            },
            "cpu_baseline": {
                "value": cpu_val,
                "unit": "verified rows/s",
                "cores": 1,
                "kind": "oracle",
                "sample": f"first {cpu_seq} of {wl.B} sequences of the same workload "
                          f"({cpu_dt:.1f} s, single thread numpy/Python)",
            },
            "e2e": {
                "value": world * rows_per_step / (e2e_ms * 1e-3),
                "unit": "verified rows/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
            },
            "gpu_launches": args.steps * (3 if args.config == "filter" else 1),
            "clocks": clocks.summary(),
        }
        if modes is not None:
            result["modes"] = modes
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------------ the draft-length gate

GATE_TEXT = ("draft-length gate + calibration update, B=1024 sequences x 5 drafted positions, "
             "6 confidence buckets seeded with the page's match table")
# the page's calibration table (PocketLLM dspark.md): bucket edges and the
# pooled match counts per confidence bucket
GATE_EDGES = [-0.5, 0.5, 1.5, 3.0, 6.0]
GATE_TOTAL = [5.0, 17.0, 19.0, 19.0, 14.0, 36.0]
GATE_HITS = [1.0, 11.0, 15.0, 17.0, 14.0, 36.0]


def gate_inputs(B=1024, K=5, seed=0x5eed0006):
    """Seeded confidences and the accepted lengths their match law implies."""
    rng = np.random.default_rng(seed)
    conf = rng.normal(2.0, 3.0, size=(B, K)).astype(np.float32)
    p = np.array(GATE_HITS) / np.array(GATE_TOTAL)
    edges = np.array(GATE_EDGES, dtype=np.float32)
    bucket = (conf[..., None] >= edges).sum(-1)
    match = rng.random((B, K)) < p[bucket]
    n_acc = np.where(match.all(1), K, match.argmin(1)).astype(np.int32)
    return conf, edges, n_acc


def run_gate(args):
    """One step = the gate for a batch, then one calibration update (two
    one-CTA launches); latency-bound, reported against HBM for the record."""
    import torch

    import oracle
    import speculative_decoding_verification_decode_gb300 as sv
    from speculative_decoding_verification_decode_gb300._build import build

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build()
    sv.load_library()
    conf_h, edges_h, nacc_h = gate_inputs(seed=0x5eed0006 + 1000 * rank)
    B, K = conf_h.shape
    conf = torch.from_numpy(conf_h).to(dev)
    edges = torch.from_numpy(edges_h).to(dev)
    nacc = torch.from_numpy(nacc_h).to(dev)
    hits = torch.tensor(GATE_HITS, dtype=torch.float64, device=dev)
    total = torch.tensor(GATE_TOTAL, dtype=torch.float64, device=dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():  # as for the verification workloads: L2 left holding clean lines
        flush_w.fill_(1)
        flush_r.sum()

    def step(c, e, na, h, t):
        # the update clamps each accepted length to the submitted one
        g = sv.gate_draft_lengths(c, e, h, t)
        sv.gate_update(c, g.n_submit, na, e, h, t, decay=1.0)
        return g

    for _ in range(args.warmup):
        flush()
        step(conf, edges, nacc, hits, total)
    torch.cuda.synchronize(dev)
    # the step is two tiny launches: capture it in a CUDA graph so the timed
    # region holds the GPU work, not the host's launch overhead
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(conf, edges, nacc, hits, total)
        with torch.cuda.graph(graph, stream=side):
            g = step(conf, edges, nacc, hits, total)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms_local = float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)]))
    ms = max_over_ranks(ms_local, dist, dev)
    # end to end: confidences and lengths from pinned host memory, lengths back
    conf_p, nacc_p = torch.from_numpy(conf_h).pin_memory(), torch.from_numpy(nacc_h).pin_memory()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 20))
    e_s.record(stream)
    for _ in range(e2e_steps):
        c = conf_p.to(dev, non_blocking=True)
        na = nacc_p.to(dev, non_blocking=True)
        out = step(c, edges, na, hits, total).cu_k.to("cpu", non_blocking=True)
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, dist, dev)
    result = None
    if rank == 0:
        peak, peak_kind = measured_peak_gbs()
        nb = len(GATE_TOTAL)
        moved = 2 * B * K * 4 + 4 * B * 4 + 4 * nb * 8 + (nb - 1) * 8  # conf twice, lengths, table
        t0 = time.perf_counter()
        prm = oracle.GateParams()
        n_o, _ = oracle.gate_batch(conf_h, None, None, edges_h, np.array(GATE_HITS), np.array(GATE_TOTAL), prm)
        oracle.update_table(conf_h, n_o, np.minimum(nacc_h, n_o), edges_h, np.array(GATE_HITS),
                            np.array(GATE_TOTAL), 1.0)  # (the kernel clamps the same way)
        cpu_dt = time.perf_counter() - t0
        result = {
            "metric": "gated sequences/s (draft-length gate and calibration update)",
            "value": world * B / (ms * 1e-3),
            "unit": "sequences/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f64",
            "data": "synthetic (seeded; the page's calibration table)",
            "config": {"workload": f"gate: {GATE_TEXT}", "B": B, "K": K, "launch": "CUDA graph per step",
                       "l2": "flushed between timed steps (512 MB write, then a 512 MB read)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": "gate_kernel + update_kernel (one CTA each)",
                         "achieved": moved / (ms_local * 1e-3) / 1e9, "peak": peak,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst)", "unit": "GB/s",
                         "frac": moved / (ms_local * 1e-3) / 1e9 / peak, "traffic": None,
                         "note": "launch-latency bound: a few KB per step"},
            "cpu_baseline": {"value": B / cpu_dt, "unit": "sequences/s", "cores": 1, "kind": "oracle",
                             "sample": f"the whole batch of {B} sequences ({cpu_dt:.2f} s, single thread Python)"},
            "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": "sequences/s",
                    "h2d_bytes_per_step": B * K * 4 + B * 4, "d2h_bytes_per_step": (B + 1) * 4,
                    "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,  # one graph of two kernels per step
            "clocks": clocks.summary(),
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------------ the decoding loop

DECODER_TEXT = ("speculative decoding rounds (draft 5, verify, commit) as one CUDA graph, B=64, "
                "V=128256 bf16 logits from a synthetic table model, temperature 0.8")


class _TableModel:
    """Synthetic next-token logits: a table row picked by a hash of the last
    two tokens (no trained weights exist here)."""

    def __init__(self, torch, dev, V, H, seed, dtype):
        g = torch.Generator().manual_seed(seed)
        self.table = (torch.randn(H, V, generator=g) * 3.0).to(device=dev, dtype=dtype)
        self.H, self.torch, self.dev = H, torch, dev

    def next_logits(self, tokens, lengths):
        torch = self.torch
        rows = torch.arange(tokens.shape[0], device=self.dev)
        t1 = tokens[rows, (lengths.long() - 1).clamp(min=0)].long()
        t2 = tokens[rows, (lengths.long() - 2).clamp(min=0)].long()
        return self.table[(t1 * 1000003 + t2 * 7919) % self.H]

    def rows(self, tokens, lengths, k):
        return self.torch.stack([self.next_logits(tokens, lengths + j) for j in range(k + 1)], dim=1)


LMHEAD_TEXT = ("verification from hidden states: B=64 K=5 V=128256 d=4096, bf16 states and projection, "
               "T=0.8 rejection sampling; logits = H W^T on the tensor cores, then the logits verification")


def measured_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


def run_lmhead(args):
    """One step = the LM head over every verified position (target and draft
    states) and the verification of those logits (a memset and two launches).
    The product dominates: it is reported against the tensor-core peak."""
    import torch

    import speculative_decoding_verification_decode_gb300 as sv
    from speculative_decoding_verification_decode_gb300._build import build
    from workloads.lm_head import make_lm_head

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build()
    sv.load_library()
    wl = make_lm_head(seed=0x5EED0007 + 1000 * rank)
    B, K, V, d = wl.B, wl.K, wl.V, wl.d
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    ht, hd, w = bf(wl.h_target), bf(wl.h_draft), bf(wl.w)
    T = torch.from_numpy(wl.temperature).to(dev)
    tok = torch.from_numpy(wl.tokens).to(dev)
    u = torch.from_numpy(wl.uniforms).to(dev)
    ws = sv.lm_head_workspace(B, B * K, V, dev)
    stream = torch.cuda.current_stream(dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1)
        flush_r.sum()

    step = lambda i: sv.lm_head_verify(ht, hd, w, T, tok, u, workspace=ws)
    for i in range(args.warmup):
        flush()
        r = step(i)
    torch.cuda.synchronize(dev)
    n_acc = r.n_accepted.cpu().numpy()
    barrier(dist, dev)
    with ClockSampler(local, args.clocks_csv) as clocks:
        per_step = timed_steps(torch, stream, args.steps, flush, step)
    barrier(dist, dev)
    ms_local = float(np.mean(per_step))
    ms = max_over_ranks(ms_local, dist, dev)
    # the product alone (the roofline's kernel) over the same 704 rows, into
    # the same workspace rows (target rows and draft rows are contiguous there)
    ldv = (V + 3) // 4 * 4
    rows = B * (2 * K + 1)
    hall = torch.cat([ht, hd])
    lall = ws[256:256 + rows * ldv * 4].view(torch.float32).view(-1, ldv)[:, :V]
    prod_ms = float(np.mean(timed_steps(torch, stream, args.steps, flush,
                                        lambda i: sv.lm_head_logits(hall, w, out=lall))))
    # end to end: states, tokens, uniforms and temperatures from pinned host
    # memory (the projection is a resident weight), results back
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hth = pin(wl.h_target.view(np.int16)).view(torch.bfloat16)
    hdh = pin(wl.h_draft.view(np.int16)).view(torch.bfloat16)
    Th, tokh, uh = pin(wl.temperature), pin(wl.tokens), pin(wl.uniforms)
    h2d = sum(x.numel() * x.element_size() for x in (hth, hdh, Th, tokh, uh))
    for _ in range(2):
        sv.lm_head_verify(hth, hdh, w, Th, tokh, uh, workspace=ws)
    torch.cuda.synchronize(dev)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 20))
    e_s.record(stream)
    for _ in range(e2e_steps):
        rr = sv.lm_head_verify(hth, hdh, w, Th, tokh, uh, workspace=ws)
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, dist, dev)
    assert np.array_equal(rr.n_accepted.numpy(), n_acc)
    result = None
    if rank == 0:
        import oracle
        burst, sustained, kind = measured_peak_tflops()
        flops = 2.0 * rows * V * d
        achieved = flops / (prod_ms * 1e-3) / 1e12
        t0 = time.perf_counter()
        oracle.accept_lm_head(wl.h_target[:K + 1], wl.h_draft[:K], wl.w, "bf16", wl.temperature[:1],
                              wl.tokens[:K], wl.uniforms[:K + 1], 1, K)
        cpu_dt = time.perf_counter() - t0
        result = {
            "metric": METRIC,
            "value": world * B * (K + 1) / (ms * 1e-3),
            "unit": "verified rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded Philox states and projection, random-init)",
            "config": {
                "workload": f"lmhead: {LMHEAD_TEXT}",
                "B": B, "K": K, "V": V, "d": d,
                "us_per_round": ms * 1e3,
                "rounds_per_s": world * B / (ms * 1e-3),
                "mean_accepted": float(n_acc.mean()),
                "product_us": prod_ms * 1e3,
                "verify_us": (ms_local - prod_ms) * 1e3,
                "product_flops_per_step": flops,
                "l2": "flushed between timed steps (512 MB write, then a 512 MB read)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            },
            "roofline": {
                "bound": "tensor",
                "kernel": "svl::lm_head_kernel",
                "achieved": achieved,
                "peak": sustained,
                "peak_kind": f"{kind} (MEASURED_PEAKS.json bf16_tflops_sustained; burst {burst})",
                "unit": "TFLOP/s",
                "frac": achieved / sustained,
                "frac_of_burst": achieved / burst,
                "traffic": None,
            },
            "cpu_baseline": {
                "value": (K + 1) / cpu_dt,
                "unit": "verified rows/s",
                "cores": 1,
                "kind": "oracle",
                "sample": f"one sequence of the same workload ({cpu_dt:.1f} s, fp64 numpy products "
                          "then the Python verification)",
            },
            "e2e": {
                "value": world * B * (K + 1) / (e2e_ms * 1e-3),
                "unit": "verified rows/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 3 * B * 4,
                "ms_per_step": e2e_ms,
            },
            "gpu_launches": args.steps * 2,
            "clocks": clocks.summary(),
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


def run_decoder(args):
    """One step = one speculative decoding round of the whole batch, replayed
    from a CUDA graph; the metric counts committed tokens."""
    import torch

    import speculative_decoding_verification_decode_gb300 as sv
    from speculative_decoding_verification_decode_gb300._build import build
    from speculative_decoding_verification_decode_gb300.decoder import SpeculativeDecoder

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build()
    sv.load_library()
    B, K, V, H = 64, 5, 128256, 509
    rounds = args.warmup + args.steps
    target = _TableModel(torch, dev, V, H, seed=31 + rank, dtype=torch.bfloat16)
    draft = _TableModel(torch, dev, V, H, seed=31 + rank, dtype=torch.bfloat16)
    draft.table = (draft.table.float() + torch.randn(draft.table.shape, device=dev) * 1.5).to(torch.bfloat16)
    L = 3 + (rounds + 2) * (K + 1)
    tok = torch.zeros(B, L, dtype=torch.int32, device=dev)
    tok[:, :3] = torch.randint(0, V, (B, 3), device=dev, dtype=torch.int32)
    lens = torch.full((B,), 3, dtype=torch.int32, device=dev)
    T = torch.full((B,), 0.8, dtype=torch.float32, device=dev)
    dec = SpeculativeDecoder(draft.next_logits, target.rows, tok, lens, K, V, temperature=T, seed=rank)
    dec.capture()
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        dec.graph.replay()
    torch.cuda.synchronize(dev)
    l0 = int(dec.lengths.sum())
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            starts[i].record(stream)
            dec.graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    committed = int(dec.lengths.sum()) - l0
    ms_local = float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)]))
    ms = max_over_ranks(ms_local, dist, dev)
    result = None
    if rank == 0:
        peak, peak_kind = measured_peak_gbs()
        tok_per_round = committed / args.steps
        # bytes of the round's verification inputs: target rows + draft rows, bf16
        moved = B * ((K + 1) + K) * V * 2
        result = {
            "metric": "committed tokens/s (speculative decoding rounds, synthetic table model)",
            "value": world * tok_per_round / (ms * 1e-3),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded table model; no trained weights)",
            "config": {"workload": f"decoder: {DECODER_TEXT}", "B": B, "K": K, "V": V,
                       "tokens_per_round": tok_per_round, "launch": "CUDA graph per round",
                       "l2": "not flushed: each round's rows are freshly written by the model",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": "whole round (model gathers, softmax draws, verify)",
                         "achieved": moved / (ms_local * 1e-3) / 1e9, "peak": peak,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst)", "unit": "GB/s",
                         "frac": moved / (ms_local * 1e-3) / 1e9 / peak, "traffic": None,
                         "note": "bytes = the verification inputs a round produces; the table model's "
                                 "own gathers and the drafter's softmax draws are extra"},
            "cpu_baseline": None,
            "e2e": None,
            "gpu_launches": None,
            "clocks": clocks.summary(),
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


def run_reference(args):
    """The CPU oracle timed on the host cores (the reference arm of this repo)."""
    import workloads

    rank, world, _ = dist_info()
    if rank != 0:
        return None
    wl = make_workload(args.config)
    per_step = []
    for i in range(args.warmup + args.steps):
        v, nseq, dt = oracle_rows_per_s(wl, budget_s=args.ref_step_budget)
        if i >= args.warmup:
            per_step.append((v, nseq, dt))
    value = float(np.mean([v for v, _, _ in per_step]))
    nseq = per_step[-1][1]
    seqs_per_step = 1 if args.config == "latency1" else wl.B  # latency1: a step is one B=1 round
    ms = float(np.mean([dt / n for _, n, dt in per_step])) * seqs_per_step * 1e3
    result = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "verified rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded Philox; shapes and distributions of the workload)",
        "config": {"workload": f"{args.config}: {CONFIG_TEXT[args.config]}", "B": seqs_per_step,
                   "K": wl.K, "V": wl.V, "input_dtype": wl.dtype},
        "cpu_baseline": {"value": value, "unit": "verified rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: the first {nseq} of {wl.B} sequences "
                                   f"(bounded to {args.ref_step_budget:.0f} s of CPU work)"},
        "e2e": {"value": value, "unit": "verified rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="config2", choices=list(CONFIG_TEXT) + ["gate", "decoder", "lmhead"],
                    help="a verification workload, 'gate' for the draft-length gate, or 'decoder' "
                         "for whole speculative decoding rounds")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline field")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the SM clock samples of the timed region in this file")
    ap.add_argument("--no-modes", action="store_true",
                    help="config2 only: skip the greedy and single-sequence summaries")
    ap.add_argument("--ref-step-budget", type=float, default=6.0,
                    help="seconds of oracle work per step of the reference arm")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.config == "decoder":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "no reference decoding loop: the "
                              "oracle verifies single steps"}), flush=True)
            return None
        return run_decoder(args)
    if args.config == "lmhead":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the LM head's reference is the oracle's "
                              "fp64 product; its time is the lmhead line's cpu_baseline"}), flush=True)
            return None
        return run_lmhead(args)
    if args.config == "gate":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the gate's reference is the oracle; "
                              "its time is the gate line's cpu_baseline"}), flush=True)
            return None
        return run_gate(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
