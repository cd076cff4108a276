"""Benchmark of the quantisation hot path on one GB300 (or N replicas).

One step is one pass of every step of the path over the full-size synthetic
workload, through the library's public API:

  * dual-layout NVFP4 + Four-Over-Six of a 256-expert MoE layer:
    gate_up bf16 [256, 4096, 6144] and down bf16 [256, 6144, 2048]
    (slice amax, rowwise and columnwise codes/scales from one read);
  * DQ(Q(w)) of both rowwise copies, written transposed as bf16 for dgrad;
  * per-token NVFP4 + Four-Over-Six of activations [16384, 6144] and
    [32768, 2048];
  * NF4 (blocksize 64) of gate_up, the routed union of an 8192-token top-8
    Zipf(1.1) router and the dequant of only the routed experts.

The metric is algorithmic GB/s: every input read once and every output
written once (bf16 2 B/elem, NVFP4 0.5 + 1/16 B/elem per layout, NF4
0.5 + 4/64 B/elem, bf16 dequant out 2 B/elem, plus the small per-slice /
per-token FP32 scales and router indices), divided by the device time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
With --gpus N > 1 (launched by torch.distributed.run) every rank runs the
same step on its own GPU (replicas: the path has no exchange step); value is
the sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "moe_layer_256x(4096x6144,6144x2048)+act(16384x6144,32768x2048)+nf4_routed(8192x8,zipf1.1)"
METRIC = "quantize/dequant GB/s and % of GB300 HBM peak (NVFP4 dual+4/6, NF4 routed)"

GATE_UP = (256, 4096, 6144)
DOWN = (256, 6144, 2048)


def set_experts(n):
    """Reduces the expert count (profiling of small cases only)."""
    global GATE_UP, DOWN
    GATE_UP = (n, GATE_UP[1], GATE_UP[2])
    DOWN = (n, DOWN[1], DOWN[2])
ACTS = ((16384, 6144), (32768, 2048))
TOKENS, TOPK = 8192, 8


def nvfp4_bytes(n):           # one NVFP4 layout out
    return n // 2 + n // 16


def nf4_bytes(n):
    return n // 2 + (n // 64) * 4


# --------------------------------------------------------------- workload

class Workload:
    def __init__(self, device, seed_base=1):
        import torch
        from rl_nvfp4_quantize_gb300 import synth
        self.dev = device
        E, R, K = GATE_UP
        self.gu = synth.expert_weights(*GATE_UP, seed=seed_base + 1, device=device)
        self.dn = synth.expert_weights(*DOWN, seed=seed_base + 2, device=device)
        self.x = [synth.activations(T, H, seed=seed_base + 3 + i, device=device)
                  for i, (T, H) in enumerate(ACTS)]
        self.topk = synth.zipf_router(TOKENS, E, TOPK, seed=seed_base + 5, device=device)
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16

        def e(shape, dt):
            return torch.empty(shape, dtype=dt, device=device)

        def dual_out(shape):
            n, r, k = shape
            return dict(codes_row=e((n, r, k // 2), u8), scales_row=e((n, r, k // 16), u8),
                        codes_col=e((n, k, r // 2), u8), scales_col=e((n, k, r // 16), u8),
                        amax=e((n,), f32), tensor_scale=e((n,), f32))
        self.q_gu = dual_out(GATE_UP)
        self.q_dn = dual_out(DOWN)
        self.dqt_gu = e((E, K, R), bf)
        self.dqt_dn = e((DOWN[0], DOWN[2], DOWN[1]), bf)
        self.q_x = [dict(codes=e((T, H // 2), u8), scales=e((T, H // 16), u8), token_scale=e((T,), f32))
                    for T, H in ACTS]
        self.nf4 = dict(codes=e((E, R, K // 2), u8), absmax=e((E, R, K // 64), f32))
        self.nf4_dst = e(GATE_UP, bf)
        self.hit = e((E,), torch.int32)
        self.nhit = e((1,), torch.int32)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def calls(self):
        """(name, callable, algorithmic bytes, kernel launches) for one step."""
        import torch
        import rl_nvfp4_quantize_gb300 as nvq
        n_gu = GATE_UP[0] * GATE_UP[1] * GATE_UP[2]
        n_dn = DOWN[0] * DOWN[1] * DOWN[2]

        def dual_launches(E, R, K):
            # zeroing of amax and the arrival counters, the single pass over
            # the stack, the tensor scales
            return 3
        L = []
        for name, w, q, n, E in (("nvfp4_quantize_dual[gate_up]", self.gu, self.q_gu, n_gu, GATE_UP[0]),
                                 ("nvfp4_quantize_dual[down]", self.dn, self.q_dn, n_dn, DOWN[0])):
            L.append((name, (lambda w=w, q=q: nvq.nvfp4_quantize_dual(
                w, four_over_six=True, status=self.status, out=q)),
                2 * n + 2 * nvfp4_bytes(n) + 8 * E, dual_launches(*w.shape)))
        for name, q, dst, n, E in (("nvfp4_dequant_t[gate_up]", self.q_gu, self.dqt_gu, n_gu, GATE_UP[0]),
                                   ("nvfp4_dequant_t[down]", self.q_dn, self.dqt_dn, n_dn, DOWN[0])):
            L.append((name, (lambda q=q, dst=dst: nvq.nvfp4_dequant_t(
                q["codes_row"], q["scales_row"], q["tensor_scale"], out=dst)),
                nvfp4_bytes(n) + 2 * n + 4 * E, 1))
        for i, (T, H) in enumerate(ACTS):
            L.append(("act_quantize_per_token[%dx%d]" % (T, H), (lambda i=i: nvq.act_quantize_per_token(
                self.x[i], four_over_six=True, status=self.status, out=self.q_x[i])),
                2 * T * H + nvfp4_bytes(T * H) + 4 * T, 1))
        L.append(("nf4_quantize[gate_up]", lambda: nvq.nf4_quantize(self.gu, status=self.status, out=self.nf4),
                  2 * n_gu + nf4_bytes(n_gu), 1))
        L.append(("nf4_dequant_routed[gate_up]", lambda: nvq.nf4_dequant_routed(
            self.nf4["codes"], self.nf4["absmax"], self.topk, dst=self.nf4_dst, status=self.status,
            hit_list=self.hit, n_hit=self.nhit), None, 2))
        return L

    def routed_bytes(self):
        """Algorithmic bytes of the routed dequant: only the hit experts."""
        E, R, K = GATE_UP
        nh = int(self.nhit.item())
        per = R * K
        return nh * (nf4_bytes(per) + 2 * per) + TOKENS * TOPK * 4 + 4 * (E + 1)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.rows:
            if ts < t0 - 0.2 or ts > t1 + 0.2:
                continue
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- the oracle

def synth_module():
    """The seeded input generators (synth.py), loaded from their file alone:
    the CPU arms use them without importing the package, which loads the
    CUDA library."""
    import importlib.util
    path = os.path.join(ROOT, "rl_nvfp4_quantize_gb300", "synth.py")
    spec = importlib.util.spec_from_file_location("nvq_synth_standalone", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def host_info():
    """The host the CPU baseline ran on: its logical CPUs and CPU model."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:  # lscpu missing: fall back to /proc/cpuinfo
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"host_cpus": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


def host_sample(frac, wl=None, seed_base=1):
    """Host (CPU) inputs for a proportional sample of the step: a fraction
    `frac` of the rows of each weight stack (taken from expert 0) and of the
    tokens of each activation tensor.  Taken from the device workload when
    given, else generated on the host with the same distributions."""
    r_gu = max(16, int(round(frac * GATE_UP[0] * GATE_UP[1])) // 16 * 16)
    r_dn = max(16, int(round(frac * DOWN[0] * DOWN[1])) // 16 * 16)
    assert r_gu <= GATE_UP[1] and r_dn <= DOWN[1], "sample larger than one expert"
    toks = [max(1, int(round(frac * T))) for T, _ in ACTS]
    if wl is not None:
        gu = wl.gu[0:1, :r_gu].cpu()
        dn = wl.dn[0:1, :r_dn].cpu()
        xs = [wl.x[i][:t].cpu() for i, t in enumerate(toks)]
    else:
        synth = synth_module()
        gu = synth.expert_weights(1, r_gu, GATE_UP[2], seed=seed_base + 1)
        dn = synth.expert_weights(1, r_dn, DOWN[2], seed=seed_base + 2)
        xs = [synth.activations(t, H, seed=seed_base + 3 + i) for i, (t, (_, H)) in enumerate(zip(toks, ACTS))]
    return gu, dn, xs


def oracle_step(gu, dn, xs):
    """One pass of the oracle over a host sample (same calls as a GPU step:
    both-layout NVFP4 + Four-Over-Six with the slice amax, transposed
    dequant, per-token activations, NF4 quantise and dequant).  Returns
    (algorithmic bytes, seconds, description, elements)."""
    import numpy as np
    import torch
    import oracle

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    total_b, secs, parts, elems = 0, 0.0, [], 0
    for name, w in (("gate_up", gu), ("down", dn)):
        r, K = w.shape[1], w.shape[2]
        x = u16(w)
        t0 = time.perf_counter()
        o = oracle.nvfp4_quantize(x, four_over_six=True)
        oracle.nvfp4_quantize_colwise(x, four_over_six=True)
        oracle.nvfp4_dequant_t(o["codes"], o["scales"], o["G"], r, K)
        secs += time.perf_counter() - t0
        n = r * K
        total_b += 2 * n + 2 * nvfp4_bytes(n) + nvfp4_bytes(n) + 2 * n
        elems += 2 * n
        parts.append("%s[0,:%d,:]" % (name, r))
    for i, x in enumerate(xs):
        t, H = x.shape
        t0 = time.perf_counter()
        oracle.act_quantize_per_token(u16(x), four_over_six=True)
        secs += time.perf_counter() - t0
        total_b += 2 * t * H + nvfp4_bytes(t * H) + 4 * t
        elems += t * H
        parts.append("act[:%d,:%d]" % (t, H))
    r, K = gu.shape[1], gu.shape[2]
    t0 = time.perf_counter()
    q = oracle.nf4_quantize(u16(gu))
    oracle.nf4_dequant(q["codes"], q["absmax"], 1, r, K)
    secs += time.perf_counter() - t0
    n = r * K
    total_b += 2 * n + nf4_bytes(n) + nf4_bytes(n) + 2 * n
    elems += 2 * n
    parts.append("nf4 gate_up[0,:%d,:]" % r)
    return total_b, secs, ", ".join(parts), elems


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, timed on the host on
    a bounded proportional sample of the same workload per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    frac = args.ref_frac
    gu, dn, xs = host_sample(frac)
    for _ in range(args.warmup):
        oracle_step(gu, dn, xs)
    tot_b, tot_s, desc = 0, 0.0, ""
    for _ in range(args.steps):
        b, sec, desc, _ = oracle_step(gu, dn, xs)
        tot_b += b
        tot_s += sec
    value = tot_b / tot_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_fraction": frac},
            "cpu_baseline": dict({"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": "%s per step (fraction %g of the step)" % (desc, frac)},
                                 **host_info()),
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------- main

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def setup_dist(args, backend="nccl"):
    """Rank, world size and local rank from the torchrun environment; with
    more than one rank, joins the process group (NCCL on the GPU machine; the
    host tests use gloo) and selects this rank's GPU."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    """The largest value of v over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, bytes_per_step, steps, elapsed_max):
    """Whole-job GB/s: every rank runs the same step on its own GPU (weak
    scaling), so the job moves world * bytes_per_step per step, and the job
    takes as long as its slowest rank."""
    return world * bytes_per_step * steps / elapsed_max / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-frac", type=float, default=1.0 / 512)
    ap.add_argument("--experts", type=int, default=256,
                    help="experts per weight stack (256 = the full layer; fewer only for profiling)")
    ap.add_argument("--only", default=None,
                    help="run only the calls whose name contains this text (profiling)")
    ap.add_argument("--ref-frac", type=float, default=1.0 / 8192)
    ap.add_argument("--no-context", action="store_true",
                    help="skip the context measurements outside the step")
    ap.add_argument("--unfused", action="store_true",
                    help="with --case: also time the dequant + per-expert cuBLAS comparison")
    ap.add_argument("--case", default=None, choices=["dgrad", "nf4_linear", "mxfp8", "nest"],
                    help="run one context measurement alone on a reduced case (profiling)")
    ap.add_argument("--tokens", type=int, default=2048,
                    help="router tokens of --case")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.experts != 256:
        set_experts(args.experts)
    if args.impl == "reference":
        # the CPU oracle alone: the product's CUDA library is neither built
        # nor loaded on this arm
        run_reference(args)
        return
    if args.case:
        import __graft_entry__
        __graft_entry__.build()
        run_case(args)
        return

    import __graft_entry__
    __graft_entry__.build()

    import torch
    import rl_nvfp4_quantize_gb300 as nvq  # noqa: F401
    world, rank, local = setup_dist(args)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    wl = Workload(dev)
    calls = wl.calls()
    if args.only:
        calls = [c for c in calls if args.only in c[0]]
    launches_per_step = sum(c[3] for c in calls)

    for _ in range(args.warmup):
        for _, fn, _, _ in calls:
            fn()
    torch.cuda.synchronize()
    routed_b = wl.routed_bytes()
    calls = [(n, f, (b if b is not None else routed_b), k) for n, f, b, k in calls]
    step_bytes = sum(c[2] for c in calls)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for s in range(args.steps):
        for j, (_, fn, _, _) in enumerate(calls):
            ev[s][j][0].record(stream)
            fn()
            ev[s][j][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed_max = max_over_ranks(world, elapsed)
    ms_step = 1e3 * elapsed_max / args.steps
    value = job_rate(world, step_bytes, args.steps, elapsed_max)

    per_call = []
    for j, (name, _, b, k) in enumerate(calls):
        times = [ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(args.steps)]
        per_call.append((name, statistics.mean(times), b, statistics.median(times)))
    peak, peak_src = load_peaks()
    dom = max(per_call, key=lambda x: x[1])
    dom_gbs = dom[2] / (dom[1] / 1e3) / 1e9
    elems = call_elements(wl)
    breakdown = {}
    for n, ms, b, med in per_call:
        e = {"ms": round(ms, 4), "ms_median": round(med, 4), "GB/s": round(b / (ms / 1e3) / 1e9, 1),
             "frac": round(b / (ms / 1e3) / 1e9 / peak, 4)}
        if n in elems:
            e["Gelem/s"] = round(elems[n] / (ms / 1e3) / 1e9, 2)
        dram = load_traffic(n)
        if dram:
            e["dram_over_algorithmic"] = round(dram / b, 3)
        sec = load_sectors(n)
        if sec:
            e["sectors"] = sec
        breakdown[n] = e
    st = int(wl.status.item())
    n_routed = int(wl.nhit.item())  # of the timed steps' router (the context reuses the buffer)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(wl, calls, 10, stream, world)

    context = None
    if not args.no_context:
        context = measure_context(wl, dev, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b, sec, desc, el = oracle_step(*host_sample(args.cpu_frac, wl))
        cpu = {"value": round(b / sec / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "%s: fraction %g of one step, %.1f s single-threaded"
                         % (desc, args.cpu_frac, sec),
               "elem_per_s": round(el / sec, 1),
               "extrapolated_step_s": round(step_bytes / (b / sec), 1)}
        cpu.update(host_info())

    traffic = load_traffic(dom[0])
    issue = issue_view(dom[0], dom[1], GATE_UP if "gate_up" in dom[0] else DOWN)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "gate_up": list(GATE_UP), "down": list(DOWN),
                   "activations": [list(a) for a in ACTS], "router": [TOKENS, TOPK, "zipf1.1"],
                   "four_over_six": True, "l2": "inputs larger than L2 (gate_up 12.9 GB)",
                   "routed_experts": n_routed, "step_bytes": step_bytes,
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"kernel": dom[0], "bound": "hbm", "achieved": round(dom_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(dom_gbs / peak, 4), "traffic": traffic,
                     "peak_source": peak_src, "issue": issue},
        "hbm_frac_step": round(value / world / peak, 4),
        "breakdown": breakdown,
        "gpu_launches": launches_per_step * args.steps,
        "status_word": st,
        "clocks": sampler.summary(wall0, wall1),
        "context": context,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def call_elements(wl):
    """Elements each step call processes (input elements; for the routed
    dequant the elements of the hit experts)."""
    n_gu = GATE_UP[0] * GATE_UP[1] * GATE_UP[2]
    n_dn = DOWN[0] * DOWN[1] * DOWN[2]
    out = {"nvfp4_quantize_dual[gate_up]": n_gu, "nvfp4_quantize_dual[down]": n_dn,
           "nvfp4_dequant_t[gate_up]": n_gu, "nvfp4_dequant_t[down]": n_dn,
           "nf4_quantize[gate_up]": n_gu,
           "nf4_dequant_routed[gate_up]": int(wl.nhit.item()) * GATE_UP[1] * GATE_UP[2]}
    for T, H in ACTS:
        out["act_quantize_per_token[%dx%d]" % (T, H)] = T * H
    return out


# Instruction issue peak of the GPU: 152 SMs x 4 schedulers x one warp
# instruction (32 threads) per cycle at the 2070 MHz maximum SM clock.
ISSUE_PEAK = 152 * 4 * 32 * 2.07e9


def issue_view(kernel_name, ms, shape):
    """The dominant call seen as instruction-issue bound: executed thread
    instructions per second (instructions per element from the committed ncu
    capture x elements per second measured here) against ISSUE_PEAK."""
    ipe = load_profile_table().get("_instr_per_elem", {}).get(kernel_name)
    if not ipe:
        return None
    n = shape[0] * shape[1] * shape[2]
    achieved = ipe * n / (ms / 1e3)
    return {"bound": "issue", "instr_per_elem": ipe, "achieved": round(achieved / 1e12, 2),
            "peak": round(ISSUE_PEAK / 1e12, 2), "unit": "Tinstr/s",
            "frac": round(achieved / ISSUE_PEAK, 4)}


def load_profile_table():
    """The committed per-call ncu figures (profiles/traffic.json), or {}."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        return d if isinstance(d, dict) else {}
    except (OSError, ValueError):
        return {}


def load_traffic(kernel_name):
    """DRAM bytes per call of an entry point from the committed ncu capture of
    the current kernels on the full-size workload; None for any other size."""
    if GATE_UP[0] != 256:
        return None
    v = load_profile_table().get(kernel_name)
    return v if isinstance(v, (int, float)) else None


def load_sectors(kernel_name):
    """Sector efficiency of a call's global loads and stores (useful bytes per
    32-byte sector moved between L1 and L2) from the committed ncu capture."""
    v = load_profile_table().get("_sectors", {}).get(kernel_name)
    return v if isinstance(v, dict) else None


def cuda_timed(fn, reps):
    """Mean device time of one call in ms: three warm-up calls, then `reps`
    calls between two CUDA events on the current stream."""
    import torch
    for _ in range(3):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def measure_context(wl, dev, peak):
    """Measurements outside the step (not part of `value`): the small
    configurations and the routing savings at small token counts.
      * one bf16 weight [512, 256], no Four-Over-Six: quantise + dequantise,
        launch-bound, in microseconds per pair of calls;
      * dual-layout NVFP4 + Four-Over-Six of a 32-expert gate_up stack
        [32, 4096, 6144] (the first 32 slices of the layer's stack), the
        rowwise-only quantisation (with and without Four-Over-Six) and the
        rowwise dequantisation of the same stack;
      * routed NF4 dequant for 8, 32 and 128 tokens of the same top-8 Zipf(1.1)
        router: how many of the 256 experts are hit and what that costs."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    from rl_nvfp4_quantize_gb300 import synth

    timed = cuda_timed
    out = {}
    w1 = synth.single_weight(device=dev)
    q1 = nvq.nvfp4_quantize(w1, four_over_six=False)
    dq1 = nvq.nvfp4_dequant(q1["codes"], q1["scales"], q1["tensor_scale"])

    def small():
        nvq.nvfp4_quantize(w1, four_over_six=False, out=q1)
        nvq.nvfp4_dequant(q1["codes"], q1["scales"], q1["tensor_scale"], out=dq1)
    api_us = 1e3 * timed(small, 200)
    # the same launches replayed from a CUDA graph: device time without the
    # Python binding's per-call overhead
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        small()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        small()
    out["single_weight_512x256_quant+dequant_us"] = {
        "python_api": round(api_us, 2), "cuda_graph": round(1e3 * timed(graph.replay, 200), 2)}
    E, R, K = min(32, GATE_UP[0]), GATE_UP[1], GATE_UP[2]
    q32 = {k: v[:E] for k, v in wl.q_gu.items()}
    n = E * R * K
    ms = timed(lambda: nvq.nvfp4_quantize_dual(wl.gu[:E], four_over_six=True, out=q32), 5)
    gbs = (2 * n + 2 * nvfp4_bytes(n) + 8 * E) / (ms / 1e3) / 1e9
    out["dual_%dx%dx%d" % (E, R, K)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                        "frac": round(gbs / peak, 4)}
    # rowwise-only quantisation (with and without Four-Over-Six) and the
    # rowwise dequantisation of the same stack
    qr = {"codes": q32["codes_row"], "scales": q32["scales_row"], "amax": q32["amax"],
          "tensor_scale": q32["tensor_scale"]}
    for f46 in (False, True):  # Four-Over-Six last: the buffers end as the dual call left them
        ms = timed(lambda: nvq.nvfp4_quantize(wl.gu[:E], four_over_six=f46, out=qr), 5)
        gbs = (2 * n + nvfp4_bytes(n) + 8 * E) / (ms / 1e3) / 1e9
        out["rowwise%s_%dx%dx%d" % ("_4over6" if f46 else "", E, R, K)] = {
            "ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
    dq = torch.empty((E, R, K), dtype=torch.bfloat16, device=dev)
    ms = timed(lambda: nvq.nvfp4_dequant(qr["codes"], qr["scales"], qr["tensor_scale"], out=dq), 5)
    gbs = (nvfp4_bytes(n) + 2 * n + 4 * E) / (ms / 1e3) / 1e9
    out["dequant_%dx%dx%d" % (E, R, K)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                           "frac": round(gbs / peak, 4)}
    del dq
    routed = {}
    per = R * K
    for T in (8, 32, 128):
        topk = synth.zipf_router(T, GATE_UP[0], TOPK, seed=20 + T, device=dev)
        ms = timed(lambda: nvq.nf4_dequant_routed(wl.nf4["codes"], wl.nf4["absmax"], topk,
                                                  dst=wl.nf4_dst, hit_list=wl.hit, n_hit=wl.nhit), 10)
        nh = int(wl.nhit.item())
        b = nh * (nf4_bytes(per) + 2 * per) + T * TOPK * 4 + 4 * (GATE_UP[0] + 1)
        routed["tokens=%d" % T] = {"experts_hit": nh, "ms": round(ms, 4),
                                   "GB/s": round(b / (ms / 1e3) / 1e9, 1)}
    out["nf4_dequant_routed"] = routed
    stacks = {"gate_up": (wl.q_gu["codes_row"], wl.q_gu["scales_row"], wl.q_gu["tensor_scale"], GATE_UP),
              "down": (wl.q_dn["codes_row"], wl.q_dn["scales_row"], wl.q_dn["tensor_scale"], DOWN)}
    out["nvfp4_dgrad"] = measure_dgrad(stacks, wl.topk, dev)
    out["nf4_routed_linear"] = measure_nf4_linear(
        {"gate_up": (wl.nf4["codes"], wl.nf4["absmax"], GATE_UP)}, wl.topk, dev)
    out["swizzled_scales"] = measure_swizzled(wl, dev, peak)
    out["mxfp8"] = measure_mxfp8(wl, peak)
    out["nf4_absmax_nested"] = measure_nest(wl, peak)
    return out


def measure_nest(wl, peak):
    """The nested (double-quantised) NF4 absmax of the whole gate_up
    stack's absmax, [256, 4096 x 6144 / 64] FP32: nf4_absmax_nest (4 B in;
    1 B code + 4/256 B block maximum out per value) and nf4_absmax_unnest
    (the reverse)."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    a = wl.nf4["absmax"]
    E = a.shape[0]
    n = a.numel() // E
    nb = (n + 255) // 256
    nest = nvq.nf4_absmax_nest(a)
    ms = cuda_timed(lambda: nvq.nf4_absmax_nest(a, out=nest), 5)
    b = 4 * E * n + E * n + 4 * E * nb + 4 * E
    res = {"nest_%dx%d" % (E, n): {"ms": round(ms, 4), "GB/s": round(b / (ms / 1e3) / 1e9, 1),
                                   "frac": round(b / (ms / 1e3) / 1e9 / peak, 4)}}
    dst = torch.empty((E, n), dtype=torch.float32, device=a.device)
    ms = cuda_timed(lambda: nvq.nf4_absmax_unnest(nest["codes"], nest["c1"], nest["mean"], out=dst), 5)
    res["unnest_%dx%d" % (E, n)] = {"ms": round(ms, 4), "GB/s": round(b / (ms / 1e3) / 1e9, 1),
                                    "frac": round(b / (ms / 1e3) / 1e9 / peak, 4)}
    del nest, dst
    torch.cuda.empty_cache()
    return res


def measure_mxfp8(wl, peak):
    """MXFP8 of the 32-expert gate_up stack [32, 4096, 6144]:
    rowwise only (bf16 in 2 B, codes 1 B + scales 1/32 B per element) and
    rowwise + columnwise from one read (2 + 2 x (1 + 1/32) B per element), and
    the dequantisation of the rowwise copy (1 + 1/32 B in, 2 B out)."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    E, R, K = min(32, GATE_UP[0]), GATE_UP[1], GATE_UP[2]
    n = E * R * K
    w = wl.gu[:E]
    res = {}
    q = nvq.mxfp8_quantize(w, columnwise=True)
    for name, col, b in (("mxfp8_quantize_rowwise", False, 2 * n + n + n // 32),
                         ("mxfp8_quantize_dual", True, 2 * n + 2 * (n + n // 32))):
        o = q if col else {"codes_row": q["codes_row"], "scales_row": q["scales_row"]}
        ms = cuda_timed(lambda: nvq.mxfp8_quantize(w, columnwise=col, out=o), 5)
        gbs = b / (ms / 1e3) / 1e9
        res["%s_%dx%dx%d" % (name, E, R, K)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                                 "frac": round(gbs / peak, 4)}
    d = torch.empty((E, R, K), dtype=torch.bfloat16, device=w.device)
    ms = cuda_timed(lambda: nvq.mxfp8_dequant(q["codes_row"], q["scales_row"], out=d), 5)
    gbs = (n + n // 32 + 2 * n) / (ms / 1e3) / 1e9
    res["mxfp8_dequant_%dx%dx%d" % (E, R, K)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                                  "frac": round(gbs / peak, 4)}
    del q, d
    torch.cuda.empty_cache()
    return res


def measure_swizzled(wl, dev, peak):
    """Block scales in the tensor-core tiled layout: the dual quantisation of
    the 32-expert gate_up stack and the per-token quantisation of the
    [16384, 6144] activations with tiled scales (against the same calls with
    linear scales), and the NVFP4 GEMM of cuBLASLt (torch._scaled_mm) fed
    those outputs directly -- X [16384, 6144] x W_0^T, W_0 = [4096, 6144] --
    as context for the layout's consumer (a library GEMM, not this
    library's kernel)."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    res = {}
    E, R, K = min(32, GATE_UP[0]), GATE_UP[1], GATE_UP[2]
    n = E * R * K
    w = wl.gu[:E]
    lin = {k: v[:E] for k, v in wl.q_gu.items()}
    sw = nvq.nvfp4_quantize_dual(w, four_over_six=True, swizzled_scales=True)
    for name, o, flag in (("dual_linear", lin, False), ("dual_swizzled", sw, True)):
        ms = cuda_timed(lambda: nvq.nvfp4_quantize_dual(w, four_over_six=True, out=o,
                                                        swizzled_scales=flag), 5)
        gbs = (2 * n + 2 * nvfp4_bytes(n) + 8 * E) / (ms / 1e3) / 1e9
        res[name + "_%dx%dx%d" % (E, R, K)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                                "frac": round(gbs / peak, 4)}
    T, H = ACTS[0]
    x = wl.x[0]
    qx = nvq.act_quantize_per_token(x, four_over_six=True, swizzled_scales=True)
    ms = cuda_timed(lambda: nvq.act_quantize_per_token(x, four_over_six=True, out=qx,
                                                       swizzled_scales=True), 10)
    gbs = (2 * T * H + nvfp4_bytes(T * H) + 4 * T) / (ms / 1e3) / 1e9
    res["act_swizzled_%dx%d" % (T, H)] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                          "frac": round(gbs / peak, 4)}
    if hasattr(torch, "float4_e2m1fn_x2") and H == K:
        fp4, fp8 = torch.float4_e2m1fn_x2, torch.float8_e4m3fn
        a, sa = qx["codes"].view(fp4), qx["scales"].view(fp8)
        b, sb = sw["codes_row"][0].view(fp4).t(), sw["scales_row"][0].view(fp8)
        try:
            ms = cuda_timed(lambda: torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16), 10)
            res["cublas_nvfp4_gemm_%dx%dx%d" % (T, R, K)] = {
                "ms": round(ms, 4), "TFLOP/s": round(2.0 * T * R * K / (ms / 1e3) / 1e12, 1),
                "note": "cuBLASLt block-scaled FP4 GEMM reading this library's codes and tiled "
                        "scales as produced (nominal dense FP4 peak 13500 TFLOP/s)"}
        except (RuntimeError, TypeError) as e:
            res["cublas_nvfp4_gemm"] = {"unavailable": str(e).splitlines()[0][:200]}
    del sw, qx
    torch.cuda.empty_cache()
    return res


def measure_dgrad(stacks, topk, dev, unfused=True):
    """The dgrad GEMM of the layer's routed experts read straight from the
    rowwise NVFP4 copies (tensor cores, dequantisation fused into the B
    operand): dX = dY . DQ(Q(W_e)) for the tokens the router sends to each
    expert, for gate_up and down, against the measured dense bf16 peak; and
    the same product as a dequantisation to bf16 followed by one cuBLAS
    matmul per expert, for comparison."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    from rl_nvfp4_quantize_gb300 import synth
    peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        peak = float(json.load(open(p)).get("bf16_tflops", 0)) or None
    nexp = next(iter(stacks.values()))[3][0]
    counts = torch.bincount(topk.flatten().long(), minlength=nexp).cpu().tolist()
    T = sum(counts)
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    res = {}
    for name, (codes, scales, G, (E, R, K)) in stacks.items():
        dy = synth.activations(T, R, seed=41, device=dev)
        dx = torch.empty((T, K), dtype=torch.float32, device=dev)
        ms = cuda_timed(lambda: nvq.nvfp4_dgrad(dy, counts, codes, scales, G, out=dx), 5)
        flops = 2.0 * T * R * K
        tf = flops / (ms / 1e3) / 1e12
        res[name] = {"tokens": T, "ms": round(ms, 3), "TFLOP/s": round(tf, 1),
                     "bound": "tensor", "peak_bf16_TFLOP/s": peak,
                     "frac": round(tf / peak, 4) if peak else None}
        del dx
        if unfused:
            wd = torch.empty((E, R, K), dtype=torch.bfloat16, device=dev)
            dxb = torch.empty((T, K), dtype=torch.bfloat16, device=dev)

            def dequant_then_matmul():
                nvq.nvfp4_dequant(codes, scales, G, out=wd)
                for e in range(E):
                    if counts[e]:
                        torch.matmul(dy[offs[e]:offs[e + 1]], wd[e], out=dxb[offs[e]:offs[e + 1]])
            res[name]["dequant_then_cublas_ms"] = round(cuda_timed(dequant_then_matmul, 3), 3)
            del wd, dxb
        del dy
        torch.cuda.empty_cache()
    return res


def measure_nf4_linear(stacks, topk, dev, unfused=True):
    """The forward product of the routed experts read straight from their NF4
    copies (tensor cores, dequantisation fused into the B operand):
    Y = X . DQ(W_e)^T for the tokens the router sends to each expert, against
    the measured dense bf16 peak; and the same product as the routed dequant
    to bf16 followed by one cuBLAS matmul per expert, for comparison."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    from rl_nvfp4_quantize_gb300 import synth
    peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        peak = float(json.load(open(p)).get("bf16_tflops", 0)) or None
    nexp = next(iter(stacks.values()))[2][0]
    counts = torch.bincount(topk.flatten().long(), minlength=nexp).cpu().tolist()
    T = sum(counts)
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    res = {}
    for name, (codes, absmax, (E, R, K)) in stacks.items():
        x = synth.activations(T, K, seed=43, device=dev)
        y = torch.empty((T, R), dtype=torch.bfloat16, device=dev)
        ms = cuda_timed(lambda: nvq.nf4_routed_linear(x, counts, codes, absmax, out=y), 5)
        flops = 2.0 * T * R * K
        tf = flops / (ms / 1e3) / 1e12
        res[name] = {"tokens": T, "ms": round(ms, 3), "TFLOP/s": round(tf, 1),
                     "bound": "tensor", "peak_bf16_TFLOP/s": peak,
                     "frac": round(tf / peak, 4) if peak else None}
        if unfused:
            wd = torch.empty((E, R, K), dtype=torch.bfloat16, device=dev)
            hit = torch.empty((E,), dtype=torch.int32, device=dev)
            nh = torch.empty((1,), dtype=torch.int32, device=dev)

            def dequant_then_matmul():
                nvq.nf4_dequant_routed(codes, absmax, topk, dst=wd, hit_list=hit, n_hit=nh)
                for e in range(E):
                    if counts[e]:
                        torch.matmul(x[offs[e]:offs[e + 1]], wd[e].t(), out=y[offs[e]:offs[e + 1]])
            res[name]["dequant_then_cublas_ms"] = round(cuda_timed(dequant_then_matmul, 3), 3)
            del wd
        del x, y
        torch.cuda.empty_cache()
    return res


def run_case(args):
    """One context measurement alone, on a reduced expert count and router
    (the small cases the ncu captures use): --case dgrad quantises gate_up
    and down stacks of --experts slices rowwise (NVFP4, Four-Over-Six),
    --case nf4_linear quantises them to NF4; both route --tokens tokens top-8
    with the Zipf(1.1) router and time nvfp4_dgrad / nf4_routed_linear on
    both stacks (the cuBLAS comparison only with --unfused).  --case mxfp8
    times the MXFP8 calls on a gate_up stack of --experts slices; --case nest
    times the nested NF4 absmax of a gate_up stack of --experts slices.
    Prints one JSON object."""
    import torch
    import rl_nvfp4_quantize_gb300 as nvq
    from rl_nvfp4_quantize_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E = GATE_UP[0]
    if args.case == "mxfp8":
        class _W:  # the stack measure_mxfp8 reads, without the rest of the workload
            pass
        wl = _W()
        wl.gu = synth.expert_weights(*GATE_UP, seed=2, device=dev)
        peak, _ = load_peaks()
        print(json.dumps({"case": args.case, "experts": E, "result": measure_mxfp8(wl, peak)}))
        return
    if args.case == "nest":
        class _N:  # the NF4 state measure_nest reads
            pass
        wl = _N()
        wl.nf4 = nvq.nf4_quantize(synth.expert_weights(*GATE_UP, seed=2, device=dev))
        peak, _ = load_peaks()
        print(json.dumps({"case": args.case, "experts": E, "result": measure_nest(wl, peak)}))
        return
    stacks = {}
    for name, shape, seed in (("gate_up", GATE_UP, 2), ("down", DOWN, 3)):
        w = synth.expert_weights(*shape, seed=seed, device=dev)
        if args.case == "dgrad":
            q = nvq.nvfp4_quantize(w, four_over_six=True)
            stacks[name] = (q["codes"], q["scales"], q["tensor_scale"], shape)
        else:
            q = nvq.nf4_quantize(w)
            stacks[name] = (q["codes"], q["absmax"], shape)
        del w
    topk = synth.zipf_router(args.tokens, E, TOPK, seed=6, device=dev)
    if args.case == "dgrad":
        res = measure_dgrad(stacks, topk, dev, unfused=args.unfused)
    else:
        res = measure_nf4_linear(stacks, topk, dev, unfused=args.unfused)
    print(json.dumps({"case": args.case, "experts": E, "tokens": args.tokens, "topk": TOPK,
                      "result": res}))


def measure_e2e(wl, calls, steps, stream, world):
    """Same step through the public API with the inputs in pinned host memory:
    every step copies its inputs host->device, runs the path, and copies the
    quantised results back (the bf16 dequant outputs are consumed on the
    device by the GEMMs and stay there).

    The step is cut into groups by input tensor (gate_up with its calls, down,
    each activation tensor); host->device copies, kernels and device->host
    copies run on three streams, so one group's results stream back while the
    next group's input streams in and a third group computes.  Events order
    every reuse of a device buffer across groups and steps."""
    import torch
    by_name = {c[0]: c for c in calls}

    def pick(*names):
        return [by_name[n][1] for n in names if n in by_name]
    q_out = lambda q: [q[k] for k in ("codes_row", "scales_row", "codes_col", "scales_col",
                                      "tensor_scale")]
    groups = [  # (device inputs, calls, device outputs copied back)
        ([wl.topk, wl.gu], pick("nvfp4_quantize_dual[gate_up]", "nvfp4_dequant_t[gate_up]",
                                "nf4_quantize[gate_up]", "nf4_dequant_routed[gate_up]"),
         q_out(wl.q_gu) + [wl.nf4["codes"], wl.nf4["absmax"], wl.hit, wl.nhit]),
        ([wl.dn], pick("nvfp4_quantize_dual[down]", "nvfp4_dequant_t[down]"), q_out(wl.q_dn)),
    ]
    for i, (T, H) in enumerate(ACTS):
        groups.append(([wl.x[i]], pick("act_quantize_per_token[%dx%d]" % (T, H)),
                       [wl.q_x[i]["codes"], wl.q_x[i]["scales"], wl.q_x[i]["token_scale"]]))
    groups = [g for g in groups if g[1]]
    pinned = {}

    def host(t):
        if id(t) not in pinned:
            pinned[id(t)] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        return pinned[id(t)]
    for ins, _, _ in groups:
        for d in ins:
            host(d).copy_(d)
    bi = sum(d.numel() * d.element_size() for ins, _, _ in groups for d in ins)
    bo = sum(d.numel() * d.element_size() for _, _, outs in groups for d in outs)
    step_bytes = sum(c[2] for c in calls)
    s_in, s_in2, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    inputs_free = [ev() for _ in groups]    # the group's kernels no longer read its inputs
    outputs_free = [ev() for _ in groups]   # the group's results have left the device

    def one():
        for g, (ins, fns, outs) in enumerate(groups):
            # each input crosses the link as two halves on two streams (one
            # stream alone does not fill the host-to-device link)
            s_in.wait_event(inputs_free[g])
            s_in2.wait_event(inputs_free[g])
            for d in ins:
                flat_d, flat_h = d.view(-1), host(d).view(-1)
                half = flat_d.numel() // 2
                with torch.cuda.stream(s_in):
                    flat_d[:half].copy_(flat_h[:half], non_blocking=True)
                with torch.cuda.stream(s_in2):
                    flat_d[half:].copy_(flat_h[half:], non_blocking=True)
            for si in (s_in, s_in2):
                arrived = ev()
                arrived.record(si)
                stream.wait_event(arrived)
            stream.wait_event(outputs_free[g])
            for fn in fns:
                fn()
            done = ev()
            done.record(stream)
            inputs_free[g].record(stream)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for d in outs:
                    host(d).copy_(d, non_blocking=True)
            outputs_free[g].record(s_out)
    one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    streams = (stream, s_in, s_in2, s_out)
    # the end of every step on every stream: step i ends when its last
    # stream does (steps overlap across streams, so a step's time is the
    # distance between consecutive step ends)
    ends = [[torch.cuda.Event(enable_timing=True) for _ in streams] for _ in range(steps)]
    barrier(world)
    a.record(stream)
    for si in (s_in, s_in2, s_out):
        si.wait_event(a)
    for i in range(steps):
        one()
        for e, s in zip(ends[i], streams):
            e.record(s)
    torch.cuda.synchronize()
    end_ms = [max(a.elapsed_time(e) for e in row) for row in ends]
    per_step = sorted([end_ms[0]] + [end_ms[i] - end_ms[i - 1] for i in range(1, steps)])
    el = max_over_ranks(world, end_ms[-1] / 1e3)
    return {"value": round(job_rate(world, step_bytes, steps, el), 3), "unit": "GB/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": steps, "ms_per_step": round(1e3 * el / steps, 3),
            "ms_per_step_median": round(per_step[len(per_step) // 2], 3),
            "ms_per_step_min": round(per_step[0], 3), "ms_per_step_max": round(per_step[-1], 3),
            "overlap": "host-to-device copies (two streams), kernels and device-to-host copies"}


if __name__ == "__main__":
    main()
