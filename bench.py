"""Benchmark: MoE decode tokens/s of the 30-layer routed + shared FFN stack.

Workload (default): the 30-layer decode stack at full shape (d=2816, f=704,
128 experts, top-8, shared expert f=2816, int4 affine groups of 64), every
expert resident in HBM, one token per step (B = 1) through all 30 layers,
512 synthetic tokens (bf16 N(0,1)) cycled, router logits biased by the
Zipf(s=1.1) / reuse-0.6 expert trace of the slot-cache workload.  Each step
streams 1.2 GB of expert weights, far more than the 129 MB L2, so no flush is
needed between steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (bounded sample, same metric and config).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE decode tokens/s (30-layer routed+shared FFN), % of 8 TB/s HBM roofline"
UNIT = "tokens/s"
N_LAYERS = 30
N_TOKENS = 512
SEED = 2
NOMINAL_HBM = 8e12


def _shape():
    from workload import FULL
    return FULL


def bytes_per_token_layer(sh) -> dict:
    """Algorithmic bytes of one B=1 token through one layer, per kernel kind."""
    nG_d = sh.d // 64
    gu_r = (sh.f // 8) * nG_d * 576
    gu_s = (sh.f_shared // 8) * nG_d * 576
    dn_r = (sh.d // 16) * (sh.f // 64) * 576
    dn_s = (sh.d // 16) * (sh.f_shared // 64) * 576
    router = sh.n_experts * sh.d * 2
    ffn = gu_s + dn_s + sh.top_k * (gu_r + dn_r)
    return {"router_topk_plan": router + sh.d * 2,
            "gateup_gelu_gemv": gu_s + sh.top_k * gu_r,
            "down_combine_gemv": dn_s + sh.top_k * dn_r,
            "ffn_total": ffn,
            # one launch of the single-launch kernel runs the token through every layer
            "decode_persistent": N_LAYERS * (router + ffn)}


# The kernel function a profiled kind times at the benchmark's shape (the
# clustered persistent kernel is the default single-launch decode kernel).
KERNEL_FUNCTION = {"decode_persistent": "k_decode_cluster"}


def algorithmic_bytes(bpl: dict, kind: str):
    """(FFN bytes, router bytes) of one launch of kind: the FFN bytes are the
    selected experts plus the shared expert, the router rows apart."""
    if kind == "decode_persistent":
        return N_LAYERS * bpl["ffn_total"], N_LAYERS * bpl["router_topk_plan"]
    if kind == "router_topk_plan":
        return 0, bpl[kind]
    return bpl[kind], 0


def config_dict(sh):
    return {"workload": f"decode{N_LAYERS}_resident_zipf", "layers": N_LAYERS, "tokens": N_TOKENS, "B": 1,
            "d": sh.d, "f": sh.f, "f_shared": sh.f_shared, "experts": sh.n_experts, "top_k": sh.top_k,
            "group": sh.group, "weights": "int4 affine g64, fp16 scale+bias", "residency": "all experts in HBM",
            "routing": "router logits + Zipf(1.1)/reuse-0.6 bias trace",
            "l2": "no flush: 1.2 GB of weights per step vs 129 MB L2"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources that decide each captured kernel's DRAM traffic: its translation
# unit and the headers it includes (the launch shape lives in kernels.h).
TRAFFIC_SOURCES = {
    "decode_persistent": ("decode_cluster.cu", "common.cuh", "internal.h", "kernels.h"),
}


def traffic_digest(names):
    import hashlib
    src = os.path.join(ROOT, "bit_routed_expert_router_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(names):
        with open(os.path.join(src, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, for each kernel whose
    sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] in TRAFFIC_SOURCES \
                    and parts[2] == traffic_digest(TRAFFIC_SOURCES[parts[0]]):
                out[parts[0]] = float(parts[1])
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            # the timed region starts only once the sampler is writing rows
            deadline = time.time() + 10.0
            while time.time() < deadline:
                if os.path.getsize(self.file.name) > 0:
                    break
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def mark(self, start: bool):
        """Host wall-clock bounds of the timed region (rows outside it are not counted)."""
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def result(self):
        if self.proc is None:
            return None
        try:
            with open(self.file.name) as fh:
                rows = [r.split(",") for r in fh.read().strip().splitlines() if r.strip()]
            os.unlink(self.file.name)
        except Exception:
            return None
        return clock_summary(rows, self.t0, self.t1)


def _smi_time(ts: str):
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(ts.strip(), fmt).timestamp()
        except ValueError:
            continue
    return None


def clock_summary(rows, t0=None, t1=None):
    """Median SM clock, max clock and active throttle reasons of the nvidia-smi
    rows whose timestamp lies in the timed region [t0, t1] (all rows when the
    bounds or the timestamps are missing)."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    total = 0
    for r in rows:
        r = [x.strip() for x in r]
        try:
            smv, mxv = float(r[1]), float(r[2])
        except (ValueError, IndexError):
            continue
        total += 1
        ts = _smi_time(r[9]) if len(r) > 9 else None
        if t0 is not None and t1 is not None and ts is not None and not (t0 - 0.025 <= ts <= t1 + 0.025):
            continue
        sm.append(smv)
        mx.append(mxv)
        for i, n in enumerate(names):
            if len(r) > 5 + i and r[5 + i].lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
           "samples": len(sm), "samples_total": total}
    if t0 is not None and t1 is not None:
        out["region_s"] = round(t1 - t0, 4)
        out["sm_mhz_x_s"] = round(statistics.median(sm) * (t1 - t0), 2)
    return out


def time_k_steps(run_k, stream, clk, min_seconds: float = 1.0, max_reps: int = 400):
    """Time regions of exactly K steps (run_k(rep) enqueues one region), each
    bracketed by CUDA events on the launch stream, back to back until at least
    min_seconds have passed, so the clock sampler sees the timed work.  Returns
    (seconds over all regions, regions)."""
    import math

    import torch

    def region(rep):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_k(rep)
        e1.record(stream)
        return e0, e1

    # an untimed probe region sizes the repetitions (and keeps a slow first
    # region, e.g. while the clock sampler's first queries hold the driver,
    # out of the figure)
    probe = region(0)
    probe[1].synchronize()
    t_probe = probe[0].elapsed_time(probe[1]) / 1e3
    reps = max(1, min(max_reps, int(math.ceil(min_seconds / max(t_probe, 1e-6)))))
    clk.mark(True)
    pairs = [region(r) for r in range(1, reps + 1)]
    pairs[-1][1].synchronize()
    clk.mark(False)
    return sum(a.elapsed_time(b) for a, b in pairs) / 1e3, reps


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def maybe_init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def aggregate(dist, local_seconds: float, local_units: float):
    """Max time over ranks and summed units (replicas: no data-path collective)."""
    if dist is None:
        return local_seconds, local_units
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------- oracle timing

def oracle_token_layer_seconds(layers_cpu: list, H, bias, n_samples: int, budget_s: float, threads: int = 1):
    """Time the oracle on (token, layer) samples with `threads` host threads over
    matrix rows; returns (mean seconds, samples, threads in effect)."""
    import oracle
    cores = oracle.set_threads(threads)
    lays = [oracle.Layer(w, _shape().top_k) for w in layers_cpu]
    times = []
    t_start = time.perf_counter()
    for i in range(n_samples):
        li = i % len(lays)
        t = i % H.shape[0]
        x = oracle.rmsnorm_bf16(oracle.as_bits(H[t]), 1e-6)
        b = bias[t, li] if bias is not None else None
        t0 = time.perf_counter()
        lays[li].forward(x, b)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    oracle.set_threads(1)
    return statistics.mean(times), len(times), cores


def cpu_baseline_entry(layers_cpu: list, H, bias, budget_s: float):
    """The oracle at one thread (the line's value) and at every host core (an
    extra entry), each on a bounded sample of (token, layer) evaluations,
    extrapolated to 30 layers per token."""
    mean_s, n, cores = oracle_token_layer_seconds(layers_cpu, H, bias, 64, budget_s / 2)
    mean_a, n_a, cores_a = oracle_token_layer_seconds(layers_cpu, H, bias, 64, budget_s / 2,
                                                      threads=os.cpu_count() or 1)
    return {"value": 1.0 / (N_LAYERS * mean_s), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} (token, layer) evaluations on layers 0-1, {mean_s:.2f} s each, "
                      f"extrapolated x{N_LAYERS} layers per token",
            "all_cores": {"value": 1.0 / (N_LAYERS * mean_a), "cores": cores_a,
                          "sample": f"{n_a} evaluations, {mean_a:.2f} s each, matrix rows over {cores_a} threads"}}


def gen_cpu_layers(n: int):
    """A few full-shape layers on the host (generated on the GPU when one is present)."""
    import torch
    from workload import gen_layer
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    out = []
    for layer in range(n):
        w = gen_layer(_shape(), seed=SEED, layer=layer, device=dev)
        out.append({"router_w": w["router_w"].cpu(),
                    "experts": {k: v.cpu() for k, v in w["experts"].items()},
                    "shared": {k: v.cpu() for k, v in w["shared"].items()}})
        del w
    return out


def host_inputs():
    import numpy as np
    from workload import bias_from_targets, gen_hidden, zipf_reuse_targets
    sh = _shape()
    H = gen_hidden(N_TOKENS, sh.d, seed=SEED)
    tg = zipf_reuse_targets(N_TOKENS, N_LAYERS, sh.n_experts, sh.top_k, seed=SEED)
    bias = bias_from_targets(tg, sh.n_experts).astype(np.float32)
    return H, bias


# ---------------------------------------------------------------------------- arms

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    sh = _shape()
    H, bias = host_inputs()
    layers = gen_cpu_layers(2)
    # W untimed evaluations warm the oracle; the timed sample is bounded by
    # --cpu-budget seconds so the run ends within a few minutes whatever K is
    oracle_token_layer_seconds(layers, H, bias, max(args.warmup, 1), 1e9)
    t0 = time.perf_counter()
    mean_s, n, cores = oracle_token_layer_seconds(layers, H, bias, args.steps, args.cpu_budget * 4)
    wall = time.perf_counter() - t0
    tok_s = 1.0 / (N_LAYERS * mean_s)
    sample = f"{n} (token, layer) oracle evaluations on layers 0-1, extrapolated x{N_LAYERS} layers per token"
    # the same oracle with its matrix rows over every host core, for context
    mean_a, n_a, cores_a = oracle_token_layer_seconds(layers, H, bias, args.steps, args.cpu_budget,
                                                      threads=os.cpu_count() or 1)
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": ws,
            "steps": n, "warmup": max(args.warmup, 1), "ms_per_step": wall / max(n, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(sh),
            "cpu_baseline": {"value": tok_s, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                             "all_cores": {"value": 1.0 / (N_LAYERS * mean_a), "cores": cores_a,
                                           "sample": f"{n_a} evaluations, matrix rows over {cores_a} threads"}},
            "e2e": {"value": tok_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import gen_layer

    ws, rank, local = dist_env()
    dist = maybe_init_dist(ws, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh = _shape()

    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, n_layers=N_LAYERS, prenorm=1,
                          max_tokens=32)
    st, ctx = moe.moe_create(cfg, local)
    if st != moe.MOE_OK:
        raise moe.MoeError(st, moe.moe_last_error(None))
    for layer in range(N_LAYERS):
        w = gen_layer(sh, seed=SEED, layer=layer, device=dev)
        moe.check(moe.moe_init_layer(ctx, layer, w["router_w"], w["experts"], w["shared"]), ctx)
        del w
    torch.cuda.synchronize()
    H_host, bias_host = host_inputs()
    H = H_host.to(dev)
    bias = torch.from_numpy(bias_host).to(dev)          # [T, L, E]
    out = torch.empty(1, sh.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        t = i % N_TOKENS
        s, _ = moe.moe_decode_step(ctx, H[t:t + 1], 1, 0, N_LAYERS, bias[t], out, None, None, stream)
        if s != moe.MOE_OK:
            moe.check(s, ctx)

    # warm-up
    for i in range(args.warmup):
        step(i)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    if args.timeline:
        return print_timeline(moe, ctx, step, args.warmup, raw_out=args.timeline_raw)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()

    # timed regions of exactly K decode steps each (CUDA events on the launch
    # stream), repeated back to back for at least a second so that the clock
    # record covers them
    def run_k(rep):
        for i in range(args.steps):
            step(args.warmup + rep * args.steps + i)

    with ClockSampler(local) as clk:
        elapsed, reps = time_k_steps(run_k, stream, clk, args.min_seconds)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_max, units = aggregate(dist, elapsed, float(args.steps * reps))
    value = units / t_max
    clocks = clk.result()

    # per-kernel durations (event pairs around each launch, same stream, same workload)
    n_prof = min(args.steps, 32)
    moe.check(moe.moe_profile(ctx, True), ctx)
    moe.moe_get_profile(ctx)
    for i in range(n_prof):
        step(i)
    moe.check(moe.moe_profile(ctx, False), ctx)
    _, prof = moe.moe_get_profile(ctx)
    bpl = bytes_per_token_layer(sh)
    kinds = {moe.KERNEL_KINDS[i]: {"launches": n, "ms": t} for i, (n, t) in enumerate(prof) if n}
    dom = max(kinds, key=lambda k: kinds[k]["ms"])
    dur = kinds[dom]["ms"] / kinds[dom]["launches"] / 1e3
    launches_per_step = sum(v["launches"] for v in kinds.values()) / n_prof
    peak, peak_kind = load_peaks()
    # the roofline counts the FFN bytes (selected experts + shared expert); the
    # router rows are listed apart
    ffn_launch, router_launch = algorithmic_bytes(bpl, dom)
    achieved = ffn_launch / dur / 1e9
    traffic = load_traffic().get(dom)
    shares = {k: round(v["ms"] / sum(x["ms"] for x in kinds.values()), 4) for k, v in kinds.items()}

    # end to end through the C ABI with host buffers: H2D inputs, D2H output, every step
    h_pin = H_host.pin_memory()
    b_pin = torch.from_numpy(bias_host).pin_memory()
    o_pin = torch.empty(1, sh.d, dtype=torch.bfloat16).pin_memory()
    h_dev = torch.empty(1, sh.d, dtype=torch.bfloat16, device=dev)
    b_dev = torch.empty(N_LAYERS, sh.n_experts, dtype=torch.float32, device=dev)

    def e2e_step(i):
        t = i % N_TOKENS
        h_dev.copy_(h_pin[t:t + 1], non_blocking=True)
        b_dev.copy_(b_pin[t], non_blocking=True)
        s, _ = moe.moe_decode_step(ctx, h_dev, 1, 0, N_LAYERS, b_dev, out, None, None, stream)
        if s != moe.MOE_OK:
            moe.check(s, ctx)
        o_pin.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    f1.record(stream)
    f1.synchronize()
    e2e_t, e2e_units = aggregate(dist, f0.elapsed_time(f1) / 1e3, float(args.steps))
    e2e_value = e2e_units / e2e_t

    # CPU oracle on the host cores (rank 0, one GPU only), bounded sample
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(gen_cpu_layers(2), H_host, bias_host, args.cpu_budget)

    moe.moe_destroy(ctx)
    if rank == 0:
        ffn_bytes = bpl["ffn_total"] * N_LAYERS
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "timed_repeats": reps, "warmup": args.warmup, "ms_per_step": t_max / (args.steps * reps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16xint4->f32 (router int64)",
            "data": "synthetic", "config": config_dict(sh),
            "hbm_roofline_frac_8tbs": value / ws * ffn_bytes / NOMINAL_HBM,
            "bytes_per_token": ffn_bytes,
            "roofline": {"bound": "hbm", "kernel": KERNEL_FUNCTION.get(dom, dom), "achieved": achieved,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "bytes_per_launch": ffn_launch,
                         "router_bytes_per_launch": router_launch, "avg_launch_us": dur * 1e6},
            "kernel_shares": shares,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": sh.d * 2 + N_LAYERS * sh.n_experts * 4,
                    "d2h_bytes_per_step": sh.d * 2},
            "gpu_launches": int(round(launches_per_step * args.steps * reps)),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------- prefill workload

PF_TOKENS = 4096
PF_SEED = 4


# Event columns of the clustered decode kernel's per-CTA timeline (hook 5),
# in the kernel's order; columns 24.. hold summed stage times (ns).
TIMELINE_EVENTS = ["y_seen", "x_ready", "logit_out", "logits_in", "topk_done", "routed_issue", "shared_data",
                   "routed_data", "push_last", "dn_last", "stages_done", "reduced", "issue_last", "data_last",
                   "dn_a_first", "a_wait_last", "prep_cluster_barrier", "prep_y", "prep_norm", "router_publish",
                   "topk_sorted", "bulk_issued", "ops_ready"]
TIMELINE_SUMS = ["gateup_compute", "down_compute", "down_wait_for_a", "routed_data_wait", "gateup_stages",
                 "down_stages", "shared_data_wait", "end_barrier_wait"]


def print_timeline(moe, ctx, step, first, reps=3, raw_out=None):
    """Stamp one layer (the call's third) in every CTA with %globaltimer and
    print the per-event distribution (us from the first CTA's y_seen), one
    JSON line per repetition.  Diagnostic only: the stamps cost time."""
    import numpy as np
    import torch

    for rep in range(reps):
        tl = torch.zeros(152, 32, dtype=torch.int64, device="cuda")
        moe.check(moe.moe_test_hook(ctx, moe.HOOK_TIMELINE, tl.data_ptr()), ctx)
        step(first + rep)
        moe.check(moe.moe_sync(ctx), ctx)
        moe.check(moe.moe_test_hook(ctx, moe.HOOK_TIMELINE, 0), ctx)
        t = tl.cpu().numpy().astype(np.float64)
        if raw_out:
            np.save(f"{raw_out}.rep{rep}.npy", tl.cpu().numpy())
        rows = t[t[:, 0] > 1e12]
        ref = rows[:, 0].min()
        ev = {}
        for k, name in enumerate(TIMELINE_EVENTS):
            v = rows[:, k]
            v = v[v > 0]
            if len(v):
                v = (v - ref) / 1000.0
                ev[name] = {"n": int(len(v)), "min": round(float(v.min()), 2),
                            "med": round(float(np.median(v)), 2), "max": round(float(v.max()), 2)}
        sums = {name: round(float(np.median(rows[:, 24 + k])) / (1.0 if "stages" in name else 1000.0), 2)
                for k, name in enumerate(TIMELINE_SUMS)}
        print(json.dumps({"timeline_rep": rep, "ctas": int(len(rows)), "events_us": ev,
                          "per_cta_median_sums_us_or_count": sums}), flush=True)
    return 0


def prefill_flops_per_layer(sh, T):
    """Dense FLOPs of one prefill layer: routed gate/up + down per (token, k) pair, shared per token."""
    routed = 2 * T * sh.top_k * 3 * sh.d * sh.f
    shared = 2 * T * 3 * sh.d * sh.f_shared
    return routed + shared


def prefill_config(sh):
    return {"workload": f"prefill{PF_TOKENS}_resident_mixture", "layers": N_LAYERS, "tokens": PF_TOKENS,
            "d": sh.d, "f": sh.f, "f_shared": sh.f_shared, "experts": sh.n_experts, "top_k": sh.top_k,
            "group": sh.group, "weights": "int4 affine g64, fp16 scale+bias", "residency": "all experts in HBM",
            "routing": "router logits + 50/50 uniform/Zipf(0.8) bias over a per-layer permutation",
            "matrix_path": "int4 -> fp16 tiles, tcgen05 fp16 x fp16 -> fp32",
            "l2": "no flush: 12.9 GB of weights and 0.7 GB of activations per step vs 129 MB L2"}


def load_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def run_ours_prefill(args):
    import numpy as np
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import bias_from_targets, gen_hidden, gen_layer, mixture_targets

    ws, rank, local = dist_env()
    dist = maybe_init_dist(ws, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh = _shape()
    T = PF_TOKENS
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, n_layers=N_LAYERS, prenorm=1,
                          max_tokens=T)
    st, ctx = moe.moe_create(cfg, local)
    if st != moe.MOE_OK:
        raise moe.MoeError(st, moe.moe_last_error(None))
    for layer in range(N_LAYERS):
        w = gen_layer(sh, seed=PF_SEED, layer=layer, device=dev)
        moe.check(moe.moe_init_layer(ctx, layer, w["router_w"], w["experts"], w["shared"]), ctx)
        del w
    moe.check(moe.moe_test_hook(ctx, moe.HOOK_PREFILL_TC, 1), ctx)
    H_host = gen_hidden(T, sh.d, seed=PF_SEED)
    tg = mixture_targets(T, N_LAYERS, sh.n_experts, sh.top_k, seed=PF_SEED)
    bias_host = np.ascontiguousarray(bias_from_targets(tg, sh.n_experts).astype(np.float32).transpose(1, 0, 2))
    H = H_host.to(dev)
    bias = torch.from_numpy(bias_host).to(dev)           # [L, T, E]
    out = torch.empty_like(H)
    stream = torch.cuda.current_stream()

    def step():
        moe.check(moe.moe_prefill(ctx, H, T, 0, N_LAYERS, bias, out, None, stream), ctx)

    for _ in range(args.warmup):
        step()
    moe.check(moe.moe_sync(ctx, stream), ctx)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.mark(True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        e1.synchronize()
        clk.mark(False)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    elapsed = e0.elapsed_time(e1) / 1e3
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_max, units = aggregate(dist, elapsed, float(args.steps * T))
    value = units / t_max
    clocks = clk.result()

    # per-kind durations (event pairs around the routing/grouping kernels and the four GEMMs of a layer)
    moe.check(moe.moe_profile(ctx, True), ctx)
    moe.moe_get_profile(ctx)
    step()
    moe.check(moe.moe_profile(ctx, False), ctx)
    _, prof = moe.moe_get_profile(ctx)
    kinds = {moe.KERNEL_KINDS[i]: {"launches": n, "ms": t} for i, (n, t) in enumerate(prof) if n}
    shares = {k: round(v["ms"] / sum(x["ms"] for x in kinds.values()), 4) for k, v in kinds.items()}
    g = kinds["prefill_tcgen05_gemm"]
    flops_layer = prefill_flops_per_layer(sh, T)
    dur = g["ms"] / g["launches"] / 1e3                  # one layer's four GEMM launches
    peak_burst, peak_sus, peak_kind = load_bf16_peak()
    achieved = flops_layer / dur / 1e12

    # end to end with host buffers
    h_pin = H_host.pin_memory()
    b_pin = torch.from_numpy(bias_host).pin_memory()
    o_pin = torch.empty_like(h_pin).pin_memory()
    h_dev = torch.empty_like(H)
    b_dev = torch.empty_like(bias)

    def e2e_step():
        h_dev.copy_(h_pin, non_blocking=True)
        b_dev.copy_(b_pin, non_blocking=True)
        moe.check(moe.moe_prefill(ctx, h_dev, T, 0, N_LAYERS, b_dev, out, None, stream), ctx)
        o_pin.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(1, min(args.steps, 3))
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    f1.record(stream)
    f1.synchronize()
    e2e_t, e2e_units = aggregate(dist, f0.elapsed_time(f1) / 1e3, float(n_e2e * T))

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(gen_cpu_layers(2), H_host, None, args.cpu_budget)
    moe.moe_destroy(ctx)
    if rank == 0:
        line = {
            "metric": "MoE prefill tokens/s (30-layer routed+shared FFN, T=4096)", "value": value,
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16xint4->f32 (router int64)", "data": "synthetic",
            "config": prefill_config(sh),
            "roofline": {"bound": "tensor", "kernel": "prefill_tcgen05_gemm", "achieved": achieved,
                         "peak": peak_sus, "peak_kind": f"{peak_kind} bf16 sustained (fp16 runs at the bf16 rate)",
                         "unit": "TFLOP/s", "frac": achieved / peak_sus, "traffic": None,
                         "flops_per_launch": flops_layer, "avg_launch_us": dur * 1e6},
            "kernel_shares": shares,
            "e2e": {"value": e2e_units / e2e_t, "unit": "tokens/s", "h2d_bytes_per_step": int(H.numel() * 2 + bias.numel() * 4),
                    "d2h_bytes_per_step": int(out.numel() * 2)},
            "gpu_launches": int(round(N_LAYERS * 9 * args.steps)),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------- batched decode (B = 32)

BATCH = 32


def run_ours_batched(args):
    """30-layer decode, 32 independent tokens per step, all experts resident."""
    import numpy as np
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import gen_hidden, gen_layer

    ws, rank, local = dist_env()
    dist = maybe_init_dist(ws, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh = _shape()
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, n_layers=N_LAYERS, prenorm=1,
                          max_tokens=BATCH)
    st, ctx = moe.moe_create(cfg, local)
    if st != moe.MOE_OK:
        raise moe.MoeError(st, moe.moe_last_error(None))
    for layer in range(N_LAYERS):
        w = gen_layer(sh, seed=3, layer=layer, device=dev)
        moe.check(moe.moe_init_layer(ctx, layer, w["router_w"], w["experts"], w["shared"]), ctx)
        del w
    H_host = gen_hidden(N_TOKENS, sh.d, seed=3)
    H = H_host.to(dev)
    out = torch.empty(BATCH, sh.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    n_sets = N_TOKENS // BATCH

    def step(i):
        j = (i % n_sets) * BATCH
        s_, _ = moe.moe_decode_step(ctx, H[j:j + BATCH], BATCH, 0, N_LAYERS, None, out, None, None, stream)
        moe.check(s_, ctx)

    # unique experts per layer of one step (bytes the step must read)
    ids = torch.zeros(N_LAYERS, BATCH, sh.top_k, dtype=torch.int32, device=dev)
    moe.check(moe.moe_set_debug(ctx, None, ids, None, None, N_LAYERS), ctx)
    step(0)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    moe.check(moe.moe_set_debug(ctx), ctx)
    U = [len(np.unique(ids[l].cpu().numpy())) for l in range(N_LAYERS)]
    ebytes, sbytes = moe.moe_expert_bytes(cfg), moe.moe_shared_bytes(cfg)
    step_bytes = sum(u * ebytes + sbytes for u in U)

    for i in range(args.warmup):
        step(i)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.mark(True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        e1.synchronize()
        clk.mark(False)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    t_max, units = aggregate(dist, e0.elapsed_time(e1) / 1e3, float(args.steps * BATCH))
    value = units / t_max
    clocks = clk.result()
    moe.check(moe.moe_profile(ctx, True), ctx)
    moe.moe_get_profile(ctx)
    for i in range(4):
        step(i)
    moe.check(moe.moe_profile(ctx, False), ctx)
    _, prof = moe.moe_get_profile(ctx)
    kinds = {moe.KERNEL_KINDS[i]: {"launches": n, "ms": t} for i, (n, t) in enumerate(prof) if n}
    shares = {k: round(v["ms"] / sum(x["ms"] for x in kinds.values()), 4) for k, v in kinds.items()}
    launches_per_step = sum(v["launches"] for v in kinds.values()) / 4
    dom = max(kinds, key=lambda k: kinds[k]["ms"])
    g = kinds[dom]
    if dom in ("prefill_tcgen05_gemm", "small_batch_gemv"):   # a layer's GEMMs / GEMV pair read all its weights
        dom_bytes = step_bytes / N_LAYERS
    elif dom == "gateup_gelu_gemv":        # gate + up are two thirds of each expert's bytes
        dom_bytes = step_bytes * 2 / 3 / N_LAYERS
    else:
        dom_bytes = step_bytes / 3 / N_LAYERS
    dur = g["ms"] / g["launches"] / 1e3
    peak, peak_kind = load_peaks()
    achieved = dom_bytes / dur / 1e9

    h_pin = H_host.pin_memory()
    o_pin = torch.empty(BATCH, sh.d, dtype=torch.bfloat16).pin_memory()
    h_dev = torch.empty(BATCH, sh.d, dtype=torch.bfloat16, device=dev)

    def e2e_step(i):
        j = (i % n_sets) * BATCH
        h_dev.copy_(h_pin[j:j + BATCH], non_blocking=True)
        s_, _ = moe.moe_decode_step(ctx, h_dev, BATCH, 0, N_LAYERS, None, out, None, None, stream)
        moe.check(s_, ctx)
        o_pin.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    f1.record(stream)
    f1.synchronize()
    e2e_t, e2e_units = aggregate(dist, f0.elapsed_time(f1) / 1e3, float(args.steps * BATCH))
    moe.moe_destroy(ctx)
    if rank == 0:
        line = {
            "metric": "MoE batched decode tokens/s (30-layer routed+shared FFN, B=32)", "value": value,
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16xint4->f32 (router int64)", "data": "synthetic",
            "config": {"workload": f"batched{BATCH}_decode{N_LAYERS}_resident", "layers": N_LAYERS, "B": BATCH,
                       "d": sh.d, "f": sh.f, "f_shared": sh.f_shared, "experts": sh.n_experts, "top_k": sh.top_k,
                       "unique_experts_per_layer_mean": float(np.mean(U)), "bytes_per_step": step_bytes,
                       "matrix_path": "small-batch grouped GEMVs: int4 -> fp16 mma.sync from a bulk-copy ring",
                       "l2": "no flush: 11.6 GB of weights per step vs 129 MB L2"},
            "hbm_roofline_frac_measured": value / ws / BATCH * step_bytes / (peak * 1e9),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "bytes_per_launch": dom_bytes, "avg_launch_us": dur * 1e6},
            "kernel_shares": shares,
            "e2e": {"value": e2e_units / e2e_t, "unit": "tokens/s", "h2d_bytes_per_step": BATCH * sh.d * 2,
                    "d2h_bytes_per_step": BATCH * sh.d * 2},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks, "cpu_baseline": None,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------- slot-cache (host pool) decode

def host_link_peak_gbs(dev, nbytes=1 << 30, reps=5):
    """The host link's peak for the staging roofline, measured in this run on
    one 1 GiB pinned buffer: the rate of one large pinned host -> device copy
    (CUDA events on the copying stream) and the rate of plain loads from every
    SM through the link (moe_host_read_rate: how the fused step reads its
    misses).  Returns (peak, copy rate, load rate, which one is the peak)."""
    import torch
    import bit_routed_expert_router_gb300 as moe
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    e1.record()
    e1.synchronize()
    copy_gbs = reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    st, load_gbs = moe.moe_host_read_rate(src, nbytes, reps, torch.cuda.current_stream())
    if st != moe.MOE_OK:
        load_gbs = 0.0
    del src, dst
    if load_gbs > copy_gbs:
        return load_gbs, copy_gbs, load_gbs, "plain loads from every SM over a 1 GiB pinned buffer, measured in this run"
    return copy_gbs, copy_gbs, load_gbs, "one 1 GiB pinned host-to-device copy, measured in this run"


def run_ours_pool(args):
    """30-layer B = 1 decode with the routed experts in a pinned host pool and an
    LRU slot cache per layer; one sweep over N in {8, 16, 32, 64} slots."""
    import numpy as np
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import gen_layer

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh = _shape()
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, n_layers=N_LAYERS, prenorm=1,
                          max_tokens=POOL_PREFILL_CHUNK)
    st, ctx = moe.moe_create(cfg, local)
    if st != moe.MOE_OK:
        raise moe.MoeError(st, moe.moe_last_error(None))
    for layer in range(N_LAYERS):
        w = gen_layer(sh, seed=SEED, layer=layer, device=dev)
        moe.check(moe.moe_init_layer(ctx, layer, w["router_w"], w["experts"], w["shared"], moe.MOE_HOST_POOL), ctx)
        del w
    H_host, bias_host = host_inputs()
    H = H_host.to(dev)
    bias = torch.from_numpy(bias_host).to(dev)
    out = torch.empty(1, sh.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    n_tok = min(N_TOKENS, max(args.steps, 16))
    sweeps = {}
    for name, policy, staging in (("lru", moe.MOE_CACHE_LRU, moe.MOE_STAGING_HOST),
                                  ("lfu", moe.MOE_CACHE_LFU, moe.MOE_STAGING_HOST),
                                  ("lru_device", moe.MOE_CACHE_LRU, moe.MOE_STAGING_DEVICE),
                                  ("lru_fused", moe.MOE_CACHE_LRU, moe.MOE_STAGING_FUSED)):
        sweep = sweeps.setdefault(name, {})
        for n_slots in (8, 16, 32, 64):
            moe.check(moe.moe_set_slots(ctx, n_slots), ctx)
            moe.check(moe.moe_set_staging(ctx, staging), ctx)
            moe.check(moe.moe_set_cache_policy(ctx, policy), ctx)
            for t in range(args.warmup):
                moe.check(moe.moe_decode_step(ctx, H[t:t + 1], 1, 0, N_LAYERS, bias[t], out, None, None,
                                              stream)[0], ctx)
            moe.check(moe.moe_sync(ctx, stream), ctx)
            _, s0 = moe.moe_get_stats(ctx)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(n_tok):
                t = (args.warmup + i) % N_TOKENS
                moe.check(moe.moe_decode_step(ctx, H[t:t + 1], 1, 0, N_LAYERS, bias[t], out, None, None,
                                              stream)[0], ctx)
            moe.check(moe.moe_sync(ctx, stream), ctx)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            _, s1 = moe.moe_get_stats(ctx)
            hits, misses = s1.hits - s0.hits, s1.misses - s0.misses
            staged = s1.staged_bytes - s0.staged_bytes
            sweep[str(n_slots)] = {"tokens_per_s": n_tok / dt, "hit_rate": hits / max(hits + misses, 1),
                                   "misses_per_token": misses / n_tok, "staged_bytes_per_token": staged / n_tok,
                                   "host_link_gbs": staged / dt / 1e9}
    chunked = pool_prefill_run(args, ctx, dev, stream)
    moe.moe_destroy(ctx)
    link_peak, link_copy, link_load, link_source = host_link_peak_gbs(dev)
    file_tier = None
    if args.file_dir:
        file_tier = {}
        runs = [("buffered", False, 64, 0)]
        if args.file_direct:
            runs += [("o_direct", True, 64, 0), ("o_direct_slots16", True, 16, 0),
                     ("o_direct_slots16_host64", True, 16, 64)]
        for name, direct, n_slots, n_host in runs:
            try:
                r = file_tier_run(args, H, bias, out, stream, direct, n_slots, n_host)
            except moe.MoeError as e:
                r = {"error": str(e), "dir": args.file_dir}
            file_tier[name] = r
    best = sweeps["lru_fused"]["64"]
    line = {
        "metric": "MoE decode tokens/s with a per-layer LRU slot cache over a pinned host expert pool (30 layers)",
        "value": best["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": n_tok, "warmup": args.warmup,
        "ms_per_step": 1e3 / best["tokens_per_s"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16xint4->f32 (router int64)", "data": "synthetic",
        "config": {"workload": "decode30_hostpool_lru_zipf", "layers": N_LAYERS, "B": 1, "slots_reported": 64,
                   "staging_reported": "fused (one clustered-kernel launch per token: router, slot-cache step, "
                                       "misses read from the mapped pool by the consumer warps)",
                   "routing": "router logits + Zipf(1.1)/reuse-0.6 bias trace",
                   "timing": "host wall clock around the synchronised token loop"},
        "sweep_by_slots": sweeps["lru"], "sweep_by_slots_lfu": sweeps["lfu"],
        "sweep_by_slots_device_staging": sweeps["lru_device"],
        "sweep_by_slots_fused": sweeps["lru_fused"], "file_tier": file_tier,
        "chunked_prefill": chunked,
        "roofline": {"bound": "host link", "achieved": best["host_link_gbs"], "peak": link_peak, "unit": "GB/s",
                     "frac": best["host_link_gbs"] / link_peak, "traffic": None, "peak_source": link_source,
                     "host_copy_gbs": link_copy, "host_load_gbs": link_load},
        "gpu_launches": n_tok, "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


POOL_PREFILL_CHUNK = 512


def pool_prefill_run(args, ctx, dev, stream):
    """Chunked prefill through the host pool: chunks of POOL_PREFILL_CHUNK
    tokens through the 30 layers, each layer staging the union of the chunk's
    experts once from the pinned pool (host wall clock around synchronised
    calls: the host drives the staging)."""
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import gen_hidden

    sh = _shape()
    T = POOL_PREFILL_CHUNK
    H = gen_hidden(T, sh.d, seed=SEED + 7).to(dev)
    h_out = torch.empty_like(H)
    for _ in range(args.warmup):
        moe.check(moe.moe_prefill(ctx, H, T, 0, N_LAYERS, None, h_out, None, stream), ctx)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    _, s0 = moe.moe_get_stats(ctx)
    n = 4
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        moe.check(moe.moe_prefill(ctx, H, T, 0, N_LAYERS, None, h_out, None, stream), ctx)
    moe.check(moe.moe_sync(ctx, stream), ctx)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    _, s1 = moe.moe_get_stats(ctx)
    staged = s1.staged_bytes - s0.staged_bytes
    return {"chunk_tokens": T, "layers": N_LAYERS, "chunks": n, "tokens_per_s": n * T / dt,
            "ms_per_chunk": dt / n * 1e3, "experts_staged_per_layer": staged / s1.expert_bytes / n / N_LAYERS,
            "host_link_gbs": staged / dt / 1e9}


def file_tier_run(args, H, bias, out, stream, direct, n_slots, n_host):
    """The same decode with the routed experts in an expert file instead of the
    pinned pool (MOE_FILE_POOL: a miss is read by parallel pread into pinned
    staging, or, with n_host > 0, served from / read into a pinned host tier of
    n_host records per layer): tokens/s over --file-layers layers, the file
    reads' rate.  Without O_DIRECT the reads are served from the page cache the
    file was just written through; with it they go to the device under the file."""
    import torch

    import bit_routed_expert_router_gb300 as moe
    from workload import gen_layer

    sh = _shape()
    L = args.file_layers
    cfg = moe.make_config(sh.d, sh.f, sh.f_shared, sh.n_experts, sh.top_k, n_layers=L, prenorm=1, max_tokens=1)
    st, ctx = moe.moe_create(cfg, torch.cuda.current_device())
    if st != moe.MOE_OK:
        raise moe.MoeError(st, moe.moe_last_error(None))
    path = os.path.join(args.file_dir, f"moe_experts_{os.getpid()}.bin")
    flags = moe.MOE_FILE_DIRECT if direct else 0
    try:
        moe.check(moe.moe_set_expert_file(ctx, path, args.file_threads, 0, flags), ctx)
        t0 = time.perf_counter()
        for layer in range(L):
            w = gen_layer(sh, seed=SEED, layer=layer, device="cuda")
            moe.check(moe.moe_init_layer(ctx, layer, w["router_w"], w["experts"], w["shared"], moe.MOE_FILE_POOL),
                      ctx)
            del w
        init_s = time.perf_counter() - t0
        if n_host:
            moe.check(moe.moe_set_file_cache(ctx, n_host), ctx)
        moe.check(moe.moe_set_slots(ctx, n_slots), ctx)
        for t in range(args.warmup):
            moe.check(moe.moe_decode_step(ctx, H[t:t + 1], 1, 0, L, bias[t, :L].contiguous(), out, None, None,
                                          stream)[0], ctx)
        moe.check(moe.moe_sync(ctx, stream), ctx)
        _, s0 = moe.moe_get_stats(ctx)
        n_tok = min(N_TOKENS, max(args.steps, 16))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n_tok):
            t = (args.warmup + i) % N_TOKENS
            moe.check(moe.moe_decode_step(ctx, H[t:t + 1], 1, 0, L, bias[t, :L].contiguous(), out, None, None,
                                          stream)[0], ctx)
        moe.check(moe.moe_sync(ctx, stream), ctx)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        _, s1 = moe.moe_get_stats(ctx)
        misses = s1.misses - s0.misses
        read = s1.file_read_bytes - s0.file_read_bytes
        return {"layers": L, "slots": n_slots, "host_records": n_host, "tokens_per_s": n_tok / dt,
                "us_per_layer": dt / n_tok / L * 1e6, "misses_per_token": misses / n_tok,
                "host_tier_hits_per_token": (s1.host_tier_hits - s0.host_tier_hits) / n_tok,
                "file_reads_per_token": read / s1.expert_bytes / n_tok, "file_read_gbs": read / dt / 1e9,
                "threads": args.file_threads, "dir": args.file_dir,
                "file_bytes": L * sh.n_experts * ((s1.expert_bytes + 4095) // 4096 * 4096),
                "init_write_s": init_s}
    finally:
        moe.moe_destroy(ctx)
        if os.path.exists(path):
            os.remove(path)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step timed region until this much device time has passed")
    ap.add_argument("--workload", choices=["decode", "prefill", "batched", "pool"], default="decode",
                    help="decode: the B=1 30-layer decode stack (the headline); prefill: T=4096 tokens per "
                         "step; batched: B=32 tokens per step; pool: host expert pool + LRU slot sweep")
    ap.add_argument("--layers", type=int, default=30,
                    help="layers in the stack (30 is the benchmark; fewer only for small profiler captures)")
    ap.add_argument("--file-dir", default=None,
                    help="pool: also time the expert file tier with its file in this directory")
    ap.add_argument("--file-layers", type=int, default=30, help="pool: layers of the file-tier run")
    ap.add_argument("--file-threads", type=int, default=8, help="pool: pread threads of the file-tier run")
    ap.add_argument("--file-direct", action="store_true", help="pool: time the file tier with O_DIRECT reads too")
    ap.add_argument("--timeline-raw", default=None,
                    help="with --timeline: also save each repetition's raw [152][32] event array to PREFIX.repN.npy")
    ap.add_argument("--timeline", action="store_true",
                    help="decode: print the clustered kernel's per-CTA event timeline of one layer instead of timing")
    args = ap.parse_args(argv)
    global N_LAYERS
    N_LAYERS = args.layers
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "prefill":
        return run_ours_prefill(args)
    if args.workload == "batched":
        return run_ours_batched(args)
    if args.workload == "pool":
        return run_ours_pool(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
