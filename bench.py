#!/usr/bin/env python3
"""Benchmark of the verify-and-sample step on GB300.

One step = one call of spec_verify on one round of the sample_b64 workload:
B=64, gamma=4, V=128256, bf16 logits, T=0.8, draft noise sigma=1 (Zipf(1.1)
target bias).  The call is two kernels: k_sweep_vec (online-softmax statistics
of all 2*gamma+1 logit rows, 4 KB chunks) and k_race (per CTA the batch row's
accept test, then the Gumbel-max residual/bonus draw over slices of the draw
row; the batch row's CTAs form one cluster whose first CTA merges their best
keys over distributed shared memory).  Metric: verify rounds per
second (whole job, all GPUs); the line also carries verified positions/s
(B*gamma per round).  The roofline object is the verify sweep's (HBM-bound);
the race, which takes a comparable time, is issue-bound and is reported beside
it (race_ms, its share of the step).

Timing: W untimed warm-up steps, then K steps between a barrier +
cuda.synchronize() on both sides, CUDA events on the launching stream, max over
ranks.  Inputs rotate through enough sets to exceed 4x the L2 size, so no step
reads logits the previous step left in L2.  Per-kernel times come from a
separate loop of at least 200 calls with the library's timing events, with the
SM clocks sampled during it.  The other workloads (B=1 fp32, B=256 gamma=8,
the draft-noise sweep, greedy, the fused LM heads, the round's variants) are
reported in the same line.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

For N > 1 (torchrun) every rank runs an independent replica on its own GPU
(batch rows are independent; there is no exchange step): weak scaling.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec_verify rounds/s & positions/s at B=64,γ=4,V=128256; HBM GB/s % of peak"
UNIT = "rounds/s"
WORKLOAD = dict(workload="sample_b64", B=64, gamma=4, V=128256, dtype="bf16", temperature=0.8,
                sigma=1.0, seed=1003, target="N(0,2^2)+Zipf(1.1) bias",
                draft="target+N(0,sigma^2)")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--kernel-reps", type=int, default=400,
                    help="calls of the per-kernel timing loop (at least 200)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sigma", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the greedy and fused LM-head measurements")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peaks():
    """(burst, sustained) dense bf16 TFLOP/s and where they come from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


# DRAM bytes per launch of the verify sweep from an ncu capture of the same
# workload (profiles/ holds the summary); None when the kernel changed since.
SWEEP_TRAFFIC_BYTES = 150702592  # 147.796 MB read + 2.907 MB written (ncu, one launch)
LMHEAD_PASS1_TRAFFIC_BYTES = 1580866592  # 1577.972 MB read + 2.895 MB written (ncu, one launch)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif args.impl == "ours":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU baseline / reference arm: the oracle, timed on the host cores.
# ----------------------------------------------------------------------------
def oracle_rounds_per_s(w_np, budget_s: float, rows_per_step: int = 1, max_steps=None):
    """Runs the single-threaded oracle on batch rows of the workload, one or more
    rows per step, until the time budget is used; returns (rounds/s, rows, steps, s)."""
    import oracle
    zt, zd, xt, T, B = w_np
    done_rows = steps = 0
    t0 = time.perf_counter()
    while True:
        rows = [(steps * rows_per_step + k) % B for k in range(rows_per_step)]
        rnd = (steps * rows_per_step) // B
        oracle.spec_verify(zt, zd, xt, temperature=T, seed=0, rnd=rnd, rows=rows, threads=1)
        done_rows += len(rows)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and steps >= max_steps):
            break
    return (done_rows / B) / el, done_rows, steps, el


def workload_numpy(sigma):
    import torch
    from speculative_decoding_verification_21_gb300 import workloads as wl
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.sample_b64(sigma=sigma, device=dev)
    return (wl.to_oracle(w.zt), wl.to_oracle(w.zd), w.xt.cpu().numpy(), w.temperature, w.B)


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        barrier(world)
        return
    w_np = workload_numpy(args.sigma)
    # warm-up steps (untimed), then timed steps bounded by --ref-seconds
    oracle_rounds_per_s(w_np, 0.0, max_steps=max(1, min(args.warmup, 3)))
    val, rows, steps, el = oracle_rounds_per_s(w_np, args.ref_seconds, max_steps=args.steps)
    sample = (f"{steps} steps of one batch row each ({rows} of the B=64 rows, "
              f"{rows / 64:.2f} rounds) of sample_b64 sigma={args.sigma:g}, "
              f"single-threaded, {el:.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * el / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(WORKLOAD, sigma=args.sigma),
            "positions_per_s": val * 64 * 4,
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    barrier(world)


# ----------------------------------------------------------------------------
# Our arm.
# ----------------------------------------------------------------------------
def _verify_call(L, stream, sets, tokens, counts, flags, ws, B, gamma, V, dt):
    """A spec_verify call on input set i % len(sets), round i (seed 0)."""
    import speculative_decoding_verification_21_gb300 as sv
    P = ctypes.c_void_p
    sh = P(stream.cuda_stream)
    argsets = [(P(s.zt.data_ptr()), P(s.zd.data_ptr()), P(s.xt.data_ptr()), B, gamma, V, dt,
                ctypes.c_float(s.temperature),
                None if s.row_temperature is None else P(s.row_temperature.data_ptr()))
               for s in sets]
    tail = (P(tokens.data_ptr()), P(counts.data_ptr()), None, None, None, P(flags.data_ptr()),
            P(ws.data_ptr()), ctypes.c_size_t(ws.numel()), sh)
    fn = L.spec_verify

    def call(i, h=None):
        t = tail if h is None else tail[:-1] + (h,)
        rc = fn(*argsets[i % len(argsets)], 0, i, *t)
        if rc != 0:
            raise RuntimeError(f"spec_verify failed: {sv.status_string(rc)}")
    return call


def _rotation(make, per_bytes, dev):
    """Input sets of one workload whose logits add up to at least 4x the L2."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20)
    n = max(2, -(-4 * l2 // per_bytes))
    return [make(k) for k in range(n)], l2


def measure_sampling(L, dev, stream, name, sets, B, gamma, V, dt, reps, extra_keys=None):
    """Back-to-back rounds/s of spec_verify on rotating input sets, the per-kernel
    times from the library's events (the sweep, then the race), and the HBM
    roofline of the sweep on the logit bytes."""
    import torch
    import speculative_decoding_verification_21_gb300 as sv
    tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    counts = torch.empty((B,), dtype=torch.int32, device=dev)
    flags = torch.empty((B,), dtype=torch.uint8, device=dev)
    ws = sv.alloc_workspace(B, gamma, V, 0, device=dev)
    call = _verify_call(L, stream, sets, tokens, counts, flags, ws, B, gamma, V, dt)
    kms, ms = _kernel_times(L, stream, call, 2, reps)
    hbm, kind = peaks()
    esz = 4 if dt == 0 else 2
    nbytes = B * (2 * gamma + 1) * V * esz
    gbs = nbytes / (kms[0] / 1000.0) / 1e9
    acc = 0
    for i in range(len(sets)):
        call(i)
        acc += int(counts.sum().item())
    out = {"workload": name, "B": B, "gamma": gamma, "V": V,
           "dtype": "f32" if dt == 0 else "bf16",
           "rounds_per_s": 1000.0 / ms, "positions_per_s": 1000.0 / ms * B * gamma,
           "ms_per_round": ms, "kernel_ms": {"sweep": kms[0], "k_race": kms[1]},
           "mean_accepted": acc / (len(sets) * B),
           "roofline": {"bound": "hbm", "kernel": "sweep", "achieved": gbs, "peak": hbm,
                        "peak_kind": kind, "unit": "GB/s", "frac": gbs / hbm,
                        "frac_of_8TBs": gbs / 8000.0, "algorithmic_bytes": nbytes,
                        "step_frac": nbytes / (ms / 1000.0) / 1e9 / hbm},
           "l2_policy": f"inputs rotate over {len(sets)} sets",
           "gpu_launches_per_round": 2}
    if extra_keys:
        out.update(extra_keys)
    return out


def run_ours(args):
    import torch

    import speculative_decoding_verification_21_gb300 as sv
    from speculative_decoding_verification_21_gb300 import workloads as wl

    world, rank, local = dist_setup(args)
    L = sv.load(build_if_missing=False)
    dev = torch.device("cuda", local)
    B, gamma, V = 64, 4, 128256
    seed0 = WORKLOAD["seed"]

    # input sets: rotate through >= 4x L2 of logits; each rank its own replica
    base = wl.sample_b64(sigma=args.sigma, seed=seed0 + 17 * rank, device=dev)
    set_bytes = base.logit_bytes
    sets, l2 = _rotation(lambda k: base if k == 0 else wl.sample_b64(
        sigma=args.sigma, seed=seed0 + 17 * rank + 1000 * k, device=dev), set_bytes, dev)
    nsets = len(sets)
    stream = torch.cuda.current_stream(dev)
    tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    counts = torch.empty((B,), dtype=torch.int32, device=dev)
    flags = torch.empty((B,), dtype=torch.uint8, device=dev)
    ws = sv.alloc_workspace(B, gamma, V, 0, device=dev)
    step = _verify_call(L, stream, sets, tokens, counts, flags, ws, B, gamma, V, 1)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms = start.elapsed_time(stop)
    ms = max_over_ranks(ms, world)
    rounds_per_s = world * args.steps / (ms / 1000.0)

    # per-kernel times: a separate loop of >= 200 calls with the library's events
    reps = max(200, args.kernel_reps)
    with ClockSampler(local) as kclk:
        kms, call_ms = _kernel_times(L, stream, step, 2, reps)
    kavg = {"k_sweep_vec": kms[0], "k_race": kms[1], "call": call_ms}
    # the same calls captured into one CUDA graph (no host launch cost between them)
    gms = _graph_ms(lambda h, i: step(i, h), 2 * nsets)
    hbm, peak_kind = peaks()
    sweep_bytes = B * (2 * gamma + 1) * V * 2
    sweep_gbs = sweep_bytes / (kms[0] / 1000.0) / 1e9

    # end-to-end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        fn = L.spec_verify
        P = ctypes.c_void_p
        sh = P(stream.cuda_stream)
        hz = [(s.zt.cpu().pin_memory(), s.zd.cpu().pin_memory(), s.xt.cpu().pin_memory())
              for s in sets[:2]]
        dzt, dzd, dxt = torch.empty_like(base.zt), torch.empty_like(base.zd), torch.empty_like(
            base.xt)
        htok = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
        hcnt = torch.empty((B,), dtype=torch.int32).pin_memory()
        tail = (P(tokens.data_ptr()), P(counts.data_ptr()), None, None, None,
                P(flags.data_ptr()), P(ws.data_ptr()), ctypes.c_size_t(ws.numel()), sh)
        e2e_steps = max(20, min(400, args.steps // 50))

        def e2e_step(i):
            z1, z2, x = hz[i % len(hz)]
            dzt.copy_(z1, non_blocking=True)
            dzd.copy_(z2, non_blocking=True)
            dxt.copy_(x, non_blocking=True)
            rc = fn(P(dzt.data_ptr()), P(dzd.data_ptr()), P(dxt.data_ptr()), B, gamma, V, 1,
                    ctypes.c_float(base.temperature), None, 0, i, *tail)
            if rc != 0:
                raise RuntimeError(sv.status_string(rc))
            htok.copy_(tokens, non_blocking=True)
            hcnt.copy_(counts, non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        ems = max_over_ranks(s0.elapsed_time(s1), world)
        h2d = base.logit_bytes + base.xt.numel() * 4
        d2h = tokens.numel() * 4 + counts.numel() * 4
        e2e = {"value": world * e2e_steps / (ems / 1000.0), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        w_np = (wl.to_oracle(base.zt), wl.to_oracle(base.zd), base.xt.cpu().numpy(),
                base.temperature, B)
        val, rows, steps_done, el = oracle_rounds_per_s(w_np, args.cpu_seconds)
        cpu = {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"{rows} batch rows ({rows / B:.2f} rounds) of this workload, "
                         f"single-threaded, {el:.1f} s"}

    extra = {}
    if not args.no_extra:
        del sets
        torch.cuda.empty_cache()
        extra["configs"] = measure_configs(L, dev, stream, rank, reps)
        extra["greedy"] = measure_greedy(L, dev, stream, rank)
        extra["lmhead"] = measure_lmhead(L, dev, stream, rank)
        extra["lmhead_draft"] = measure_draft(L, dev, stream, rank)
        osets = [wl.sample_b64(sigma=args.sigma, seed=seed0 + 17 * rank + 1000 * k, device=dev)
                 for k in range(nsets)]
        extra["lenience"] = measure_options(L, stream, osets, tokens, counts, flags, ws,
                                            lenience=0.5)
        extra["top_k"] = measure_options(L, stream, osets, tokens, counts, flags, ws, top_k=50)
        extra["top_p"] = measure_options(L, stream, osets, tokens, counts, flags, ws, top_p=0.9)

    if rank == 0:
        line = {
            "metric": METRIC, "value": rounds_per_s, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(WORKLOAD, sigma=args.sigma),
            "l2_policy": (f"inputs rotate over {nsets} sets of {set_bytes / 1e6:.1f} MB "
                          f"(>= 4x L2 {l2 / 2**20:.0f} MiB)"),
            "parallelism": f"replicas x{world}",
            "positions_per_s": rounds_per_s * B * gamma,
            "step_effective_gbs": sweep_bytes * args.steps / (ms / world / 1000.0) / 1e9 / world,
            "roofline": {"bound": "hbm", "kernel": "k_sweep_vec", "achieved": sweep_gbs,
                         "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": sweep_gbs / hbm, "frac_of_8TBs": sweep_gbs / 8000.0,
                         "traffic": SWEEP_TRAFFIC_BYTES, "algorithmic_bytes": sweep_bytes,
                         "timing": f"CUDA events around k_sweep_vec, {reps} calls",
                         "step_share": kms[0] / (kms[0] + kms[1])},
            "race": {"kernel": "k_race", "ms": kms[1], "step_share": kms[1] / (kms[0] + kms[1]),
                     "bound": "issue and latency (a Philox4x32-10 block per four entries)"},
            "kernel_ms": kavg,
            "graph": {"ms_per_step": gms, "rounds_per_s": 1000.0 / gms,
                      "note": f"{2 * nsets} calls captured in one CUDA graph, replayed"},
            "gpu_launches": 2 * args.steps,  # k_sweep_vec and k_race per step
            "clocks": clk.summary(),
            "clocks_kernel_loop": kclk.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)


def measure_configs(L, dev, stream, rank, reps):
    """The other sampling workloads: B=1 fp32 (launch-bound), the draft-noise
    sweep of sample_b64, and B=256 gamma=8 with per-row temperatures."""
    import torch
    from speculative_decoding_verification_21_gb300 import workloads as wl
    out = {}
    # sample_b1: B=1, gamma=4, V=32000 fp32 -- one generation of many rows, one row per set
    per = 9 * 32000 * 4
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20)
    nrow = -(-4 * l2 // per)
    big = wl.sample_b1(seed=1001 + 7 * rank, device=dev, B=nrow)
    sets = [wl.Workload("sample_b1", 1, 4, 32000, torch.float32, big.temperature,
                        big.zt[b:b + 1], big.zd[b:b + 1], big.xt[b:b + 1]) for b in range(nrow)]
    out["sample_b1"] = measure_sampling(L, dev, stream, "sample_b1", sets, 1, 4, 32000, 0, reps)
    del sets, big
    for sig in (0.25, 4.0):
        sets, _ = _rotation(lambda k: wl.sample_b64(sigma=sig, seed=1003 + 17 * rank + 1000 * k,
                                                    device=dev), 64 * 9 * 128256 * 2, dev)
        out[f"sample_b64_sigma{sig:g}"] = measure_sampling(
            L, dev, stream, f"sample_b64 sigma={sig:g}", sets, 64, 4, 128256, 1, reps,
            {"sigma": sig})
        del sets
        torch.cuda.empty_cache()
    sets, _ = _rotation(lambda k: wl.sample_b256(seed=1004 + 17 * rank + 1000 * k, device=dev),
                        256 * 17 * 152064 * 2, dev)
    out["sample_b256"] = measure_sampling(L, dev, stream, "sample_b256", sets, 256, 8, 152064, 1,
                                          max(200, reps // 2),
                                          {"note": "per-row T ~ U[0.5,1.5], sigma ~ U[0.1,3], "
                                                   "-inf on 1% of tokens in 10% of draft rows"})
    del sets
    torch.cuda.empty_cache()
    return out


def measure_options(L, stream, sets, tokens, counts, flags, ws, lenience=1.0, top_k=0,
                    top_p=1.0, reps=400):
    """spec_verify_opts on the same rotating sample_b64 sets.  Lenience l: the
    comparison u <= p/(l q) runs in the same two kernels and accepts more.
    top_k: a sweep, the threshold from the candidates at or above the k-th
    largest chunk maximum, and the race on the adjusted rows.  top_p: a sweep for
    the row maxima, the nucleus cut, the thresholded sweep and the race."""
    import torch
    from speculative_decoding_verification_21_gb300 import _lib
    P = ctypes.c_void_p
    sh = P(stream.cuda_stream)
    B, gamma, V = 64, 4, 128256

    def call(i, l, k, p):
        s = sets[i % len(sets)]
        opts = _lib.Options(l, k, p)
        rc = L.spec_verify_opts(P(s.zt.data_ptr()), P(s.zd.data_ptr()), P(s.xt.data_ptr()), B,
                                gamma, V, 1, ctypes.c_float(s.temperature), None, 0, i,
                                P(tokens.data_ptr()), P(counts.data_ptr()), None, None, None,
                                P(flags.data_ptr()), ctypes.addressof(opts), P(ws.data_ptr()),
                                ctypes.c_size_t(ws.numel()), sh)
        if rc != 0:
            raise RuntimeError(f"spec_verify_opts failed ({rc})")

    acc = {}
    for key, (l, k, p) in (("plain", (1.0, 0, 1.0)), ("variant", (lenience, top_k, top_p))):
        tot = 0
        for i in range(len(sets)):
            call(i, l, k, p)
            tot += int(counts.sum().item())
        acc[key] = tot / (len(sets) * B)
    for i in range(3):
        call(i, lenience, top_k, top_p)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(reps):
        call(i, lenience, top_k, top_p)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    out = {"workload": "sample_b64", "rounds_per_s": 1000.0 / ms, "ms_per_round": ms,
           "mean_accepted": acc["variant"], "mean_accepted_plain": acc["plain"],
           "gpu_launches_per_round": (2 if not (top_k or top_p < 1.0) else
                                      2 + (1 if top_k else 0) + (2 if top_p < 1.0 else 0))}
    if lenience != 1.0:
        out["lenience"] = lenience
    if top_p < 1.0:
        out["top_p"] = top_p
    if top_k:
        out["top_k"] = top_k
        out["note"] = ("drafts are the workload's (drawn from the unadjusted q); tokens outside "
                       "the target's top-k are rejected")
    return out


def _kernel_times(L, stream, call, nkern, reps, warm=3):
    """Average per-kernel ms of `call(i)` via the library's timing events, and
    the average ms of a whole call without events."""
    import torch
    nev = max(3, nkern + 1)  # a call marks nkern + 1 events
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * nev)(*[ctypes.c_void_p(e.cuda_event) for e in ev])
    for i in range(warm):
        call(i)
    torch.cuda.synchronize()
    acc = [0.0] * nkern
    for i in range(reps):
        L.sv_set_timing_events(ctypes.cast(arr, ctypes.c_void_p), nev)
        call(warm + i)
        L.sv_set_timing_events(None, 0)
        torch.cuda.synchronize()
        for k in range(nkern):
            acc[k] += ev[k].elapsed_time(ev[k + 1])
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(reps):
        call(warm + reps + i)
    s1.record(stream)
    torch.cuda.synchronize()
    return [a / reps for a in acc], s0.elapsed_time(s1) / reps


def _graph_ms(call_on, n, replays=20):
    """Average ms per call of `call_on(stream_handle, i)`, i = 0..n-1, captured once
    into a CUDA graph on a side stream and replayed `replays` times (no host
    launch cost between the calls)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            call_on(ctypes.c_void_p(s.cuda_stream), i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for i in range(n):
            call_on(cs, i)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (replays * n)
    del g
    return ms


def measure_greedy(L, dev, stream, rank, reps=400):
    """Greedy verify on greedy_b64 (B=64, gamma=5, V=32000, bf16); inputs rotate
    over >= 4x L2."""
    import torch
    import speculative_decoding_verification_21_gb300 as sv
    from speculative_decoding_verification_21_gb300 import workloads as wl
    B, g, V = 64, 5, 32000
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20)
    per = B * (g + 1) * V * 2
    nsets = max(2, -(-4 * l2 // per))
    sets = [wl.greedy_b64(seed=2002 + 31 * k + 7 * rank, device=dev) for k in range(nsets)]
    for s in sets:
        s.zd = None  # greedy reads target logits only
    torch.cuda.empty_cache()
    tok = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.alloc_workspace(B, g, V, 1, device=dev)
    P = ctypes.c_void_p
    sh = P(stream.cuda_stream)

    def call_on(h, i):
        s = sets[i % nsets]
        rc = L.spec_verify_greedy(P(s.zt.data_ptr()), P(s.xt.data_ptr()), B, g, V, 1,
                                  P(tok.data_ptr()), P(cnt.data_ptr()), P(ws.data_ptr()),
                                  ctypes.c_size_t(ws.numel()), h)
        if rc != 0:
            raise RuntimeError(sv.status_string(rc))

    def call(i):
        call_on(sh, i)

    kms, ms = _kernel_times(L, stream, call, 1, reps)
    gms = _graph_ms(call_on, 4 * nsets)
    hbm, kind = peaks()
    gbs = per / (kms[0] / 1000.0) / 1e9
    return {"workload": "greedy_b64", "B": B, "gamma": g, "V": V, "dtype": "bf16",
            "rounds_per_s": 1000.0 / ms, "ms_per_round": ms, "kernel_ms": {"k_greedy": kms[0]},
            "graph": {"ms_per_round": gms, "rounds_per_s": 1000.0 / gms,
                      "note": f"{4 * nsets} calls captured in one CUDA graph, replayed"},
            "roofline": {"bound": "hbm", "kernel": "k_greedy", "achieved": gbs, "peak": hbm,
                         "peak_kind": kind, "unit": "GB/s", "frac": gbs / hbm,
                         "algorithmic_bytes": per},
            "l2_policy": f"inputs rotate over {nsets} sets of {per / 1e6:.1f} MB"}


def measure_draft(L, dev, stream, rank, reps=200):
    """Draft LM head + draw of one draft position (spec_lmhead_draft) on the draft
    side of lmhead_b32: B=32, draft hidden 2048, V=128256, bf16; W_draft (525 MB)
    exceeds L2."""
    import torch
    import speculative_decoding_verification_21_gb300 as sv
    from speculative_decoding_verification_21_gb300 import workloads as wl
    B, g, V, Hd = 32, 4, 128256, 2048
    w = wl.lmhead_b32(seed=1005 + 7 * rank, device=dev)
    e = w.extra
    h = e["h_d"].reshape(B, g, Hd)[:, 0].contiguous()
    tok = torch.empty((B,), dtype=torch.int32, device=dev)
    q = torch.empty((B,), dtype=torch.float32, device=dev)
    ws = sv.alloc_workspace(B, 1, V, 3, device=dev)
    P = ctypes.c_void_p
    sh = P(stream.cuda_stream)

    def call(i):
        rc = L.spec_lmhead_draft(P(h.data_ptr()), P(e["W_d"].data_ptr()), Hd, B, V,
                                 ctypes.c_float(1.0), 0, i, i % g, P(tok.data_ptr()),
                                 P(q.data_ptr()), None, None, None, P(ws.data_ptr()),
                                 ctypes.c_size_t(ws.numel()), sh)
        if rc != 0:
            raise RuntimeError(sv.status_string(rc))

    kms, ms = _kernel_times(L, stream, call, 2, reps)
    hbm, kind = peaks()
    wbytes = 2 * V * Hd
    gbs = wbytes / (kms[0] / 1000.0) / 1e9
    return {"workload": "lmhead_b32 draft side", "B": B, "V": V, "Hd": Hd,
            "dtype": "bf16 operands, fp32 accumulate", "draws_per_s": 1000.0 / ms,
            "ms_per_draw": ms, "kernel_ms": {"k_lm_draft": kms[0], "k_lm_draft_merge": kms[1]},
            "roofline": {"bound": "hbm", "kernel": "k_lm_draft", "achieved": gbs, "peak": hbm,
                         "peak_kind": kind, "unit": "GB/s", "frac": gbs / hbm,
                         "algorithmic_bytes": wbytes},
            "gpu_launches_per_draw": 2}


def measure_lmhead(L, dev, stream, rank, reps=100):
    """Fused LM heads + verify on lmhead_b32 (B=32, gamma=4, V=128256, target
    hidden 4096, draft hidden 2048, bf16): the weights (1.58 GB) exceed L2."""
    import torch
    import speculative_decoding_verification_21_gb300 as sv
    from speculative_decoding_verification_21_gb300 import workloads as wl
    B, g, V, Ht, Hd = 32, 4, 128256, 4096, 2048
    w = wl.lmhead_b32(seed=1005 + 7 * rank, device=dev)
    e = w.extra
    tok = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    flg = torch.empty((B,), dtype=torch.uint8, device=dev)
    ws = sv.alloc_workspace(B, g, V, 2, device=dev)
    P = ctypes.c_void_p
    sh = P(stream.cuda_stream)

    def call(i):
        rc = L.spec_lmhead_verify(P(e["h_t"].data_ptr()), P(e["W_t"].data_ptr()), Ht,
                                  P(e["h_d"].data_ptr()), P(e["W_d"].data_ptr()), Hd,
                                  P(w.xt.data_ptr()), B, g, V, ctypes.c_float(1.0), 0, i,
                                  P(tok.data_ptr()), P(cnt.data_ptr()), None, None,
                                  P(flg.data_ptr()), None, P(ws.data_ptr()),
                                  ctypes.c_size_t(ws.numel()), sh)
        if rc != 0:
            raise RuntimeError(sv.status_string(rc))

    kms, ms = _kernel_times(L, stream, call, 4, reps)
    rejected = float((cnt < g).float().mean().item())  # the rest draw the bonus token

    # the same round with the draft rows' statistics from the draft step
    # (spec_lmhead_draft at each position, outside the timed region): the first
    # GEMM pass streams W_target only
    hd3 = e["h_d"].reshape(B, g, Hd)
    xt_d = torch.empty((B, g), dtype=torch.int32, device=dev)
    lse = torch.empty((B, g), dtype=torch.float32, device=dev)
    logit = torch.empty((B, g), dtype=torch.float32, device=dev)
    for i in range(g):
        o = sv.spec_lmhead_draft(hd3[:, i].contiguous(), e["W_d"], pos=i, temperature=1.0,
                                 seed=0, round=0)
        xt_d[:, i], lse[:, i], logit[:, i] = o["tokens"], o["lse"], o["logit"]

    def call_drafted(i):
        rc = L.spec_lmhead_verify_drafted(
            P(e["h_t"].data_ptr()), P(e["W_t"].data_ptr()), Ht, P(e["h_d"].data_ptr()),
            P(e["W_d"].data_ptr()), Hd, P(xt_d.data_ptr()), P(lse.data_ptr()),
            P(logit.data_ptr()), B, g, V, ctypes.c_float(1.0), 0, i, P(tok.data_ptr()),
            P(cnt.data_ptr()), None, None, P(flg.data_ptr()), None, P(ws.data_ptr()),
            ctypes.c_size_t(ws.numel()), sh)
        if rc != 0:
            raise RuntimeError(sv.status_string(rc))

    dkms, dms = _kernel_times(L, stream, call_drafted, 4, reps)
    hbm, kind = peaks()
    tb, ts, tkind = tensor_peaks()
    wbytes = 2 * V * (Ht + Hd)
    flops1 = 2.0 * V * (B * (g + 1) * Ht + B * g * Hd)
    gbs1 = wbytes / (kms[0] / 1000.0) / 1e9
    tf1 = flops1 / (kms[0] / 1000.0) / 1e12
    return {"workload": "lmhead_b32", "B": B, "gamma": g, "V": V, "Ht": Ht, "Hd": Hd,
            "dtype": "bf16 operands, fp32 accumulate",
            "rounds_per_s": 1000.0 / ms, "ms_per_round": ms,
            "kernel_ms": {"k_lm_pass1": kms[0], "k_lm_finish": kms[1], "k_lm_pass2": kms[2],
                          "k_lm_merge": kms[3]},
            "rows_rejected": rejected,
            "roofline": {"bound": "hbm", "kernel": "k_lm_pass1", "achieved": gbs1, "peak": hbm,
                         "peak_kind": kind, "unit": "GB/s", "frac": gbs1 / hbm,
                         "traffic": LMHEAD_PASS1_TRAFFIC_BYTES, "algorithmic_bytes": wbytes},
            "tensor": {"kernel": "k_lm_pass1", "achieved": tf1, "peak": tb, "peak_kind": tkind,
                       "unit": "TFLOP/s", "frac": tf1 / tb, "algorithmic_flops": flops1},
            "gpu_launches_per_round": 4,
            "drafted": {"api": "spec_lmhead_verify_drafted", "rounds_per_s": 1000.0 / dms,
                        "ms_per_round": dms,
                        "kernel_ms": {"k_lm_pass1_target": dkms[0], "k_lm_finish": dkms[1],
                                      "k_lm_pass2": dkms[2], "k_lm_merge": dkms[3]},
                        "note": "drafts, lse and logits from spec_lmhead_draft (not timed)"}}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
