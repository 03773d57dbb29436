"""Benchmark of the owner-side Muon step on GB300 (prints one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--e2e-steps E] [--no-cpu-baseline]

A step is one dmuon_step over every matrix of the workload (momentum,
Nesterov input, normalisation, 5 quintic Newton-Schulz iterations, update),
with W, G and M resident in HBM.  Metric: algorithmic TFLOP/s, counting per
matrix 5*(3 m^2 n + m^3) flops (symmetric products as one triangle), plus
matrices/s.  Inputs (83.8 GB of fp32 W/G/M for the Llama-3-8B set) are far
larger than the 129 MB L2, so no flush is needed between steps.

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample
of the same workload (one matrix per step, cycling over its distinct
shapes), on this machine's host cores.

Multi-GPU: under torchrun every rank runs the whole workload as an
independent replica (the matrices of a step are independent units; there is
no exchange step on one owner), so scaling is weak; timing is max over
ranks.  ``--gpus N`` without torchrun starts the N ranks itself.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="llama3_8b")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--e2e-readback", default="both", choices=["both", "weights", "status"],
                   help="e2e result read per step: every updated weight matrix (reported as e2e), the step's "
                        "status through dmuon_get_status (reported as e2e_status), or both")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-aux", action="store_true")
    p.add_argument("--no-gram", action="store_true")
    p.add_argument("--fp16-iters", type=int, default=0,
                   help="direct backend: leading iterations with fp16 operands (0: the library's default)")
    p.add_argument("--fused", default="auto", choices=["auto", "always", "never"],
                   help="direct backend: one launch per chunk for all products (auto: the library's rule)")
    p.add_argument("--no-split", action="store_true",
                   help="skip the per-phase breakdown (a few steps with one launch per phase)")
    p.add_argument("--tile-mode", type=int, default=0, choices=[0, 1, 2, 3],
                   help="direct backend tiles: 0 automatic, 1 single CTAs (128x256), 2 CTA pairs (256x256), "
                        "3 single CTAs (128x128)")
    p.add_argument("--dealing", default="balanced", choices=["balanced", "strided"],
                   help="work items to persistent CTAs: longest first to the least loaded, or round-robin")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return None, "fallback"


def tensor_peak():
    pk, src = measured_peaks()
    if pk:
        for key in ("bf16_tflops_sustained", "bf16_tflops"):
            if key in pk and pk[key]:
                # the products run kind::f16 with fp16 operands: nominally the same dense rate as bf16
                return float(pk[key]), "of measured (%s; fp16 and bf16 share the nominal dense rate)" % key
    return FALLBACK_BF16_TFLOPS_SUSTAINED, "of fallback (sustained bf16, 1.7 PFLOP/s)"


def apply_traffic(workload):
    """DRAM bytes per Apply launch from the committed ncu summary, scaled by
    layers processed; None unless the kernel sources and the launch planning
    (work lists and their dealing, which decide L2 reuse) are the ones
    captured."""
    import hashlib
    import re
    layers = {"llama3_8b": 32, "llama3_8b_1layer": 1}.get(workload)
    path = os.path.join(ROOT, "profiles", "ns_gemm_pair_llama3_8b_1layer.md")
    if layers is None or not os.path.exists(path):
        return None
    text = open(path).read()
    sha = re.search(r"source_sha1:\s*([0-9a-f]{40})", text)
    per = re.search(r"dram_bytes_per_layer:\s*(\d+)", text)
    if not sha or not per:
        return None
    csrc = os.path.join(ROOT, "newton_schulz_nesterov_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, f), "rb").read()
                   for f in ("ns_gemm.cu", "common.cuh", "ptx.cuh", "plan.cuh"))
    if hashlib.sha1(src).hexdigest() != sha.group(1):
        return None
    return int(per.group(1)) * layers


def fused_traffic(workload):
    """DRAM bytes per fused launch from the committed ncu summary of the
    fused kernel, None unless the kernel sources and the launch planning
    hash to the captured version and the workload is the one captured."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", "ns_fused_pair_llama3_8b.md")
    if workload != "llama3_8b" or not os.path.exists(path):
        return None
    text = open(path).read()
    sha = re.search(r"source_sha1:\s*([0-9a-f]{40})", text)
    per = re.search(r"dram_bytes_per_launch:\s*(\d+)", text)
    if not sha or not per:
        return None
    csrc = os.path.join(ROOT, "newton_schulz_nesterov_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, f), "rb").read()
                   for f in ("ns_gemm.cu", "common.cuh", "ptx.cuh", "plan.cuh"))
    if hashlib.sha1(src).hexdigest() != sha.group(1):
        return None
    return int(per.group(1))


def apply_roofline(shapes, steps, apply_ms, apply_n, peak, peak_src, pairs, step_traffic, ns_steps=5,
                   single_tiles="128x256"):
    """Roofline object of the Apply kernel from its summed CUDA-event time
    (apply_ms over apply_n launches in `steps` timed steps): achieved
    algorithmic TFLOP/s against the tensor peak, and per launch the measured
    DRAM traffic (step_traffic: one iteration's Apply over all matrices, or
    None) beside the algorithmic bytes of a launch writing X' (fp16 X read,
    Z read, X' written)."""
    from newton_schulz_nesterov_gb300 import flops
    big = [(r, c) for r, c in shapes if min(r, c) > 128 or max(r, c) > 512]   # the chunked path's matrices
    achieved = flops.apply_flops(big, ns_steps) * steps / (apply_ms / 1e3) / 1e12
    launches_per_step = apply_n / steps
    alg_bytes = sum(2 * (2 * min(r, c) * max(r, c) + min(r, c) ** 2) for r, c in big) * ns_steps / launches_per_step
    kname = ("ns_gemm_pair_kernel<Apply> (X' = Z*X, Z = aI + bA + cAA, 256x256 CTA-pair tiles)" if pairs else
             "ns_gemm_kernel<Apply> (X' = Z*X, %s tiles)" % single_tiles)
    return {"kernel": kname, "bound": "tensor",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": peak_src,
            "traffic": (step_traffic * ns_steps / launches_per_step) if step_traffic else None,
            "algorithmic_bytes": alg_bytes,
            "launches_per_step": launches_per_step,
            "avg_launch_ms": apply_ms / apply_n}


def fused_roofline(shapes, steps, fused_ms, fused_n, peak, peak_src, pairs, launch_traffic, ns_steps=5,
                   single_tiles="128x256"):
    """Roofline object of the fused Newton-Schulz kernel (every Gram, Gram2
    and Apply product of a chunk in one launch) from its summed CUDA-event
    time (fused_ms over fused_n launches in `steps` timed steps): the chunked
    matrices' algorithmic flops 5 (3 m^2 n + m^3) over that time against the
    tensor peak, and per launch the measured DRAM traffic (launch_traffic,
    or None) beside the algorithmic bytes of all its products (per
    iteration: X read and A written by the Gram, A read and Z written by the
    Gram2, Z and X read and X' written by the Apply, 2-byte elements)."""
    from newton_schulz_nesterov_gb300 import flops
    big = [(r, c) for r, c in shapes if min(r, c) > 128 or max(r, c) > 512]
    achieved = flops.algorithmic_flops(big, ns_steps) * steps / (fused_ms / 1e3) / 1e12
    launches_per_step = fused_n / steps
    per_iter = sum(2 * (3 * min(r, c) * max(r, c) + 4 * min(r, c) ** 2) for r, c in big)
    kname = ("ns_gemm_pair_kernel<Fused> (all Gram, Gram2 and Apply products of a chunk, 256x256 CTA-pair tiles)"
             if pairs else "ns_gemm_kernel<Fused> (all products of a chunk, %s tiles)" % single_tiles)
    return {"kernel": kname, "bound": "tensor",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": peak_src,
            "traffic": launch_traffic,
            "algorithmic_bytes": per_iter * ns_steps / launches_per_step,
            "launches_per_step": launches_per_step,
            "avg_launch_ms": fused_ms / fused_n}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_median": statistics.median(
                    [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()] or [0.0])}


# ------------------------------------------------------------------ oracle
CPU_SHAPE_BUDGET = 1.5e13   # algorithmic flops above which a shape is not timed on the host (~30 s)


def oracle_sample(workload):
    """The CPU baseline's sample: one matrix per distinct shape of the
    workload (the first of each), with the number of matrices of that shape,
    for timing each once and extrapolating to the whole step by count.
    Shapes above CPU_SHAPE_BUDGET flops are listed but not timed (their time
    is extrapolated from the timed shapes' flop rate).
    Returns ([(index, count, timed)], description)."""
    from newton_schulz_nesterov_gb300 import workloads, flops
    w = workloads.get(workload)
    first, count = {}, {}
    for i, sh in enumerate(w.shapes):
        first.setdefault(sh, i)
        count[sh] = count.get(sh, 0) + 1
    out = []
    for sh, i in first.items():
        out.append((i, count[sh], flops.algorithmic_flops([sh]) <= CPU_SHAPE_BUDGET))
    timed = [w.shapes[i] for i, _, t in out if t]
    desc = ("one matrix per distinct shape, timed once each: %s (of %d matrices); full step extrapolated by "
            "shape count" % (", ".join("%dx%d" % s_ for s_ in timed), len(w.shapes)))
    if any(not t for _, _, t in out):
        desc += "; not timed (rate of the timed shapes): " + ", ".join(
            "%dx%d" % w.shapes[i] for i, _, t in out if not t)
    return out, desc


def time_oracle_matrix(workload, i):
    """Seconds of one fp64 oracle Muon step of matrix i of the workload."""
    import numpy as np
    import oracle
    from newton_schulz_nesterov_gb300 import workloads
    w = workloads.get(workload)
    W, G, M = (workloads.weight(w, i).numpy(), workloads.grad(w, i, 0).numpy(), workloads.momentum(w, i).numpy())
    t0 = time.perf_counter()
    oracle.muon_step(W, G, M, lr=float(np.float32(0.02)), mu=float(np.float32(0.95)))
    return time.perf_counter() - t0


def cpu_baseline(workload):
    """The fp64 oracle as it stands on this host's cores: one matrix per
    distinct shape timed once, the rate over that sample, and the seconds of
    a whole step extrapolated by shape count."""
    from newton_schulz_nesterov_gb300 import workloads, flops
    w = workloads.get(workload)
    sample, desc = oracle_sample(workload)
    secs, fl = 0.0, 0
    per = {}
    for i, cnt, timed in sample:
        if timed:
            t = time_oracle_matrix(workload, i)
            per[i] = t
            secs += t
            fl += flops.algorithmic_flops([w.shapes[i]])
    rate = fl / secs
    full = sum(cnt * (per[i] if timed else flops.algorithmic_flops([w.shapes[i]]) / rate)
               for i, cnt, timed in sample)
    return {"value": rate / 1e12, "unit": "TFLOP/s (algorithmic)", "cores": cpu_threads(), "kind": "oracle",
            "sample": desc, "seconds": secs,
            "extrapolated": {"seconds_per_step": full, "tflops": flops.algorithmic_flops(w.shapes) / full / 1e12,
                             "how": "per-shape oracle time x number of matrices of that shape"}}


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank):
    """The fp64 oracle as the reference arm: each timed step is one matrix of
    the workload's distinct shapes, in turn (warm-up steps take the smallest),
    so the run stays within a few minutes; the rate is the sampled flops over
    the sampled time, and the full step's seconds are extrapolated by shape
    count."""
    if rank != 0:
        return
    from newton_schulz_nesterov_gb300 import workloads, flops
    w = workloads.get(args.workload)
    sample, desc = oracle_sample(args.workload)
    timed = [(i, cnt) for i, cnt, t in sample if t]
    smallest = min(timed, key=lambda ic: flops.algorithmic_flops([w.shapes[ic[0]]]))[0]
    for _ in range(args.warmup):
        time_oracle_matrix(args.workload, smallest)
    secs, fl, per = 0.0, 0, {}
    for k in range(args.steps):
        i = timed[k % len(timed)][0]
        t = time_oracle_matrix(args.workload, i)
        per.setdefault(i, []).append(t)
        secs += t
        fl += flops.algorithmic_flops([w.shapes[i]])
    value = fl / secs / 1e12
    rate = fl / secs
    full = sum(cnt * (statistics.mean(per[i]) if i in per else flops.algorithmic_flops([w.shapes[i]]) / rate)
               for i, cnt, _ in sample)
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": "muon_step_tflops", "value": value,
        "unit": "TFLOP/s (algorithmic)", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "matrices_per_s": args.steps / secs,
        "config": {"workload": args.workload, "sample": "each step one matrix, cycling over: " + desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s (algorithmic)", "cores": cores,
                         "kind": "oracle", "sample": desc,
                         "extrapolated": {"seconds_per_step": full,
                                          "how": "per-shape oracle time x number of matrices of that shape"}},
        "e2e": {"value": value, "unit": "TFLOP/s (algorithmic)", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks
def rank_workload(name, rank):
    """Rank r's own problem: the named workload's shapes with inputs drawn
    from a rank-specific seed (independent problems per rank, weak scaling)."""
    import dataclasses
    from newton_schulz_nesterov_gb300 import workloads
    w = workloads.get(name)
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 7919 * rank)


def max_over_ranks(value, world):
    """Max of a per-rank float over the process group (identity at N = 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ ours
def run_ours(args, rank, world, local_rank):
    import torch
    import newton_schulz_nesterov_gb300 as dm
    from newton_schulz_nesterov_gb300 import _build, workloads, flops

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build()
    w = rank_workload(args.workload, rank)
    n = len(w.shapes)
    shapes = list(w.shapes)
    lr, mu = 0.02, 0.95

    Ws = [workloads.weight(w, i, dev) for i in range(n)]
    Ms = [workloads.momentum(w, i, dev) for i in range(n)]
    h = dm.Handle(local_rank)
    if args.tile_mode:
        dm.dmuon_set_tile_mode(h.h, args.tile_mode)
    dm.dmuon_set_balanced_dealing(h.h, args.dealing == "balanced")
    dm.dmuon_set_fused_phases(h.h, {"auto": 2, "always": 1, "never": 0}[args.fused])
    if args.fp16_iters:
        dm.dmuon_set_fp16_iterations(h.h, args.fp16_iters)
    for step in range(w.warm_steps):
        Gw = [workloads.grad(w, i, step, dev) for i in range(n)]
        h.step(Ws, Gw, Ms, lr=lr, mu=mu)
        del Gw
    Gs = [workloads.grad(w, i, w.warm_steps, dev) for i in range(n)]
    torch.cuda.synchronize()
    resident = sum(3 * 4 * r * c for r, c in shapes)

    stream = torch.cuda.current_stream()
    wp = [t.data_ptr() for t in Ws]
    gp = [t.data_ptr() for t in Gs]
    mp = [t.data_ptr() for t in Ms]

    def one_step():
        dm.dmuon_step_ptrs(h.h, wp, gp, mp, shapes, lr, mu, 5, stream=stream)

    for _ in range(max(args.warmup, 3)):
        one_step()
    rc, _ = h.status()
    if rc != 0:
        raise RuntimeError("warm-up status %d" % rc)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- timed region (device time with CUDA events on the launch stream)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    dm.dmuon_profile_read(h.h)
    dm.dmuon_profile_enable(h.h, True)
    barrier()
    torch.cuda.synchronize()
    launches0 = dm.dmuon_launch_count(h.h)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = dm.dmuon_launch_count(h.h) - launches0
    dm.dmuon_profile_enable(h.h, False)
    prof = dm.dmuon_profile_read(h.h)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    rc, _ = h.status()
    if rc != 0:
        raise RuntimeError("timed status %d" % rc)
    ms = max_over_ranks(ms, world)
    sec = ms / 1e3
    fl = flops.algorithmic_flops(shapes)
    value = fl * args.steps * world / sec / 1e12

    # ---- dominant kernel roofline (the Z*X apply phase; tensor-bound)
    peak, peak_src = tensor_peak()
    # Each phase launches once per chunk and iteration; achieved rates divide
    # the phase's algorithmic work over the timed steps by its summed time.
    apply_ms, apply_n = prof["apply"]
    fused_ms, fused_n = prof["ns_fused"]
    summary = dm.dmuon_plan_summary(h.h)
    pairs = "pairs" in summary
    single_tiles = "128x128" if "128x128 single" in summary else "128x256"
    if fused_n:
        roofline = fused_roofline(shapes, args.steps, fused_ms, fused_n, peak, peak_src, pairs,
                                  fused_traffic(args.workload), single_tiles=single_tiles)
    elif apply_n:
        roofline = apply_roofline(shapes, args.steps, apply_ms, apply_n, peak, peak_src, pairs,
                                  apply_traffic(args.workload), single_tiles=single_tiles)
    else:
        roofline = None
    phase = {k: {"ms_per_launch": (v[0] / v[1]) if v[1] else None, "launches": v[1],
                 "ms_per_step": v[0] / args.steps}
             for k, v in prof.items() if v[1]}
    hbm_peak = FALLBACK_HBM_GBS
    pk, _ = measured_peaks()
    if pk and pk.get("hbm_gbs"):
        hbm_peak = float(pk["hbm_gbs"])
    if "momentum" in phase:   # absent when every matrix runs on the small-matrix kernel
        big = [s_ for s_ in shapes if not (min(s_) <= 128 and max(s_) <= 512)]
        mom_ms_step = prof["momentum"][0] / args.steps
        phase["momentum"]["achieved_gbs"] = flops.elementwise_bytes(big) / (mom_ms_step / 1e3) / 1e9
        phase["momentum"]["frac_of_hbm"] = phase["momentum"]["achieved_gbs"] / hbm_peak

    # ---- the same step with one launch per phase and iteration: where the
    # fused kernel's time goes, phase by phase (CUDA events per launch)
    split = None
    if fused_n and not args.no_split:
        split = phase_split(args, h, wp, gp, mp, shapes, stream, lr, mu)

    # ---- the rest of Muon.step: AdamW and clipping rooflines (HBM-bound)
    aux = None
    if args.workload == "llama3_8b" and not args.no_aux:
        aux = run_aux(args, h, Gs, stream, hbm_peak)

    # ---- the Gram-space backend on the same workload (own handle and plan)
    gram = None
    if not args.no_gram:
        gram = run_gram(args, Ws, Gs, Ms, shapes, stream, world, ms / args.steps, local_rank)

    # ---- end to end through the public API with host buffers
    e2e = e2e_status = None
    if not args.no_e2e and args.e2e_steps > 0:
        if args.e2e_readback in ("both", "weights"):
            e2e = run_e2e(args, h, Ws, Gs, Ms, shapes, fl, stream, world, weights=True)
        if args.e2e_readback in ("both", "status"):
            e2e_status = run_e2e(args, h, Ws, Gs, Ms, shapes, fl, stream, world, weights=False)
            if e2e is None:
                e2e = e2e_status

    line = {
        "metric": "muon_step_tflops", "value": value, "unit": "TFLOP/s (algorithmic)",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16/bf16", "data": "synthetic",
        "matrices_per_s": n * args.steps * world / sec,
        "dense_equiv_tflops": flops.dense_flops(shapes) * args.steps * world / sec / 1e12,
        "config": {"workload": args.workload, "matrices": n, "ns_steps": 5,
                   "resident_bytes": resident,
                   "l2": ("inputs larger than L2 (%.1f GB resident W/G/M), no flush needed" % (resident / 1e9)
                          if resident > 129e6 else
                          "inputs fit in L2 (%.1f MB resident W/G/M; a latency case, not flushed)" % (resident / 1e6)),
                   "dealing": args.dealing,
                   "operands": "fp16 in the first %s iterations, bf16 after; fp32 accumulate"
                               % (args.fp16_iters or 3),
                   "parallelism": "replicas x%d" % world if world > 1 else "single GPU"},
        "gpu_launches": launches,
        "roofline": roofline,
        "phases": phase,
        "phases_per_phase_launches": split,
        "clocks": clk,
        "e2e": e2e,
        "e2e_status": e2e_status,
        "aux": aux,
        "gram_backend": gram,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    h.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def phase_split(args, h, wp, gp, mp, shapes, stream, lr, mu):
    """A few steps with the fused launch switched off (one launch per phase
    and iteration, the same tiles and arithmetic): milliseconds per step of
    each phase by CUDA events, and the whole step, beside the fused
    headline.  The handle is left fused again."""
    import torch
    import newton_schulz_nesterov_gb300 as dm
    from newton_schulz_nesterov_gb300 import flops
    dm.dmuon_set_fused_phases(h.h, False)
    try:
        for _ in range(2):
            dm.dmuon_step_ptrs(h.h, wp, gp, mp, shapes, lr, mu, 5, stream=stream)
        dm.dmuon_profile_read(h.h)
        dm.dmuon_profile_enable(h.h, True)
        steps = 3
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            dm.dmuon_step_ptrs(h.h, wp, gp, mp, shapes, lr, mu, 5, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        dm.dmuon_profile_enable(h.h, False)
        prof = dm.dmuon_profile_read(h.h)
    finally:
        dm.dmuon_set_fused_phases(h.h, {"auto": 2, "always": 1, "never": 0}[args.fused])
    big = [(r, c) for r, c in shapes if min(r, c) > 128 or max(r, c) > 512]
    out = {"steps": steps, "ms_per_step": e0.elapsed_time(e1) / steps}
    for k, v in prof.items():
        if v[1]:
            out[k] = {"ms_per_step": v[0] / steps, "launches": v[1]}
    work = {"gram": 5 * sum(min(s_) ** 2 * max(s_) for s_ in big), "gram2": 5 * sum(min(s_) ** 3 for s_ in big),
            "apply": flops.apply_flops(big)}
    for k, fl in work.items():
        if k in out and out[k]["ms_per_step"] > 0:
            out[k]["algorithmic_tflops"] = fl / (out[k]["ms_per_step"] / 1e3) / 1e12
    return out


def run_gram(args, Ws, Gs, Ms, shapes, stream, world, direct_ms, device):
    """The same step with the Gram-space Newton-Schulz backend (restart
    before the third step), timed like the headline (CUDA events, warm-up
    first) on a handle of its own.  Reports its step time, matrices/s, its
    own algorithmic flop rate, the direct-iteration-equivalent rate (the
    headline's flop count over this time) and the speed-up over the direct
    backend measured just before."""
    import torch
    import newton_schulz_nesterov_gb300 as dm
    from newton_schulz_nesterov_gb300 import flops
    wp = [t.data_ptr() for t in Ws]
    gp = [t.data_ptr() for t in Gs]
    mp = [t.data_ptr() for t in Ms]
    h = dm.Handle(device)
    dm.dmuon_set_balanced_dealing(h.h, args.dealing == "balanced")

    def one_step():
        dm.dmuon_step_ptrs(h.h, wp, gp, mp, shapes, 0.02, 0.95, 5, stream=stream, backend="gram")

    for _ in range(max(args.warmup, 3)):
        one_step()
    if h.status()[0] != 0:
        raise RuntimeError("gram warm-up status")
    dm.dmuon_profile_read(h.h)
    dm.dmuon_profile_enable(h.h, True)
    torch.cuda.synchronize()
    l0 = dm.dmuon_launch_count(h.h)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = dm.dmuon_launch_count(h.h) - l0
    dm.dmuon_profile_enable(h.h, False)
    prof = dm.dmuon_profile_read(h.h)
    rc = h.status()[0]
    h.close()
    if rc != 0:
        raise RuntimeError("gram timed status %d" % rc)
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    gfl = flops.gram_flops(shapes, 5, (2,))
    return {
        "restarts": [2], "ms_per_step": ms,
        "matrices_per_s": len(shapes) * world / (ms / 1e3),
        "algorithmic_tflops": gfl * world / (ms / 1e3) / 1e12,
        "direct_equivalent_tflops": flops.algorithmic_flops(shapes) * world / (ms / 1e3) / 1e12,
        "speedup_vs_direct": direct_ms / ms,
        "gpu_launches": launches,
        "phases": {k: {"ms_per_step": v[0] / args.steps, "launches": v[1]} for k, v in prof.items() if v[1]},
        "parity": "tests/test_gpu_gram.py (fp64 Gram oracle, 3e-2 per matrix)",
    }


def run_aux(args, h, Gs, stream, hbm_peak):
    """AdamW over the Llama-3-8B non-Muon parameters (embeddings, LM head,
    RMSNorm weights: 1.05 G elements, 28 B each per step) and segmented
    clipping of the 224 Muon gradients (one bucket per layer; sum of squares
    4 B/element + scaling 8 B/element), timed with the library's per-launch
    CUDA events."""
    import torch
    import newton_schulz_nesterov_gb300 as dm
    dev = Gs[0].device
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    shapes = [(128256, 4096), (128256, 4096)] + [(4096,)] * 65
    P = [torch.randn(s, device=dev, generator=gen) * 0.02 for s in shapes]
    G = [torch.randn(s, device=dev, generator=gen) * 1e-3 for s in shapes]
    M = [torch.zeros(s, device=dev) for s in shapes]
    V = [torch.zeros(s, device=dev) for s in shapes]
    n_el = sum(p.numel() for p in P)
    steps = args.steps
    for t in range(1, 4):
        dm.dmuon_adamw_step(h.h, P, G, M, V, step=t, stream=stream)
    dm.dmuon_profile_read(h.h)
    dm.dmuon_profile_enable(h.h, True)
    for t in range(4, 4 + steps):
        dm.dmuon_adamw_step(h.h, P, G, M, V, step=t, stream=stream)
    torch.cuda.synchronize()
    prof = dm.dmuon_profile_read(h.h)
    adamw_ms = prof["adamw"][0] / max(1, prof["adamw"][1])
    del P, G, M, V
    buckets = [i // 7 for i in range(len(Gs))]
    gp = [g.data_ptr() for g in Gs]
    nums = [g.numel() for g in Gs]
    saved = [g.clone() for g in Gs[:7]]
    for _ in range(2):
        dm.dmuon_clip_grad_norm_ptrs(h.h, gp, nums, 1e30, buckets, 32, stats=False, stream=stream)
    dm.dmuon_profile_read(h.h)
    for _ in range(steps):   # max_norm far above the norms: sum of squares, finalise, no scaling
        dm.dmuon_clip_grad_norm_ptrs(h.h, gp, nums, 1e30, buckets, 32, stats=False, stream=stream)
    torch.cuda.synchronize()
    prof = dm.dmuon_profile_read(h.h)
    dm.dmuon_profile_enable(h.h, False)
    clip_ms = prof["clip"][0] / max(1, prof["clip"][1])
    for g, s0 in zip(Gs[:7], saved):
        assert torch.equal(g, s0)  # statistics-only clipping left the gradients unchanged
    g_el = sum(nums)
    return {
        "adamw": {"elements": n_el, "ms_per_step": adamw_ms, "bytes_per_element": 28,
                  "achieved_gbs": 28 * n_el / (adamw_ms / 1e3) / 1e9,
                  "frac_of_hbm": 28 * n_el / (adamw_ms / 1e3) / 1e9 / hbm_peak, "bound": "hbm"},
        "clip_norms": {"elements": g_el, "buckets": 32, "ms_per_call": clip_ms, "bytes_per_element": 4,
                       "achieved_gbs": 4 * g_el / (clip_ms / 1e3) / 1e9,
                       "frac_of_hbm": 4 * g_el / (clip_ms / 1e3) / 1e9 / hbm_peak, "bound": "hbm"},
    }


def step_groups(shapes, target_groups=32):
    """Contiguous groups of matrices with identical shape lists (so that all
    group calls share one plan), each about 1/target_groups of the elements:
    the smallest repeating period of the shape list, replicated."""
    n = len(shapes)
    period = n
    for p in range(1, n + 1):
        if n % p == 0 and all(shapes[i] == shapes[i % p] for i in range(n)):
            period = p
            break
    total = sum(r * c for r, c in shapes)
    per = sum(r * c for r, c in shapes[:period])
    reps = 1
    while reps * per * target_groups < total and (n // period) % (reps * 2) == 0:
        reps *= 2
    size = period * reps
    return [list(range(i, i + size)) for i in range(0, n, size)]


def host_mem_available():
    """Bytes of host memory available (MemAvailable of /proc/meminfo), or None."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def run_e2e(args, h, Ws, Gs, Ms, shapes, fl, stream, world, weights=True):
    """The same step end to end through the public API with host buffers:
    every step copies its gradients in from pinned host memory and reads the
    step's result back, inside the timed region; M stays resident as
    optimizer state.  The result read is every updated weight matrix into
    pinned host memory (weights=True), or the step's status through
    dmuon_get_status (per-matrix flags, which waits for the step; W then stays
    resident too).  The step is issued as one dmuon_step call per group of
    matrices (per layer for the Llama set) so that group g's upload (and
    group g-1's read-back) run on side streams while group g computes."""
    import torch
    import newton_schulz_nesterov_gb300 as dm
    n_mats = len(shapes)
    need = sum(g.numel() * 4 for g in Gs) + (sum(x.numel() * 4 for x in Ws) if weights else 0)
    avail = host_mem_available()
    if avail is not None and need * world * 1.25 > avail:
        # every rank pins its own copies; leave the host room rather than risk its memory
        return {"value": None, "unit": "TFLOP/s (algorithmic)",
                "skipped": "pinned host copies need %.1f GB x %d ranks, %.1f GB available"
                           % (need / 1e9, world, avail / 1e9)}
    try:
        Gh = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in Gs]
        Wh = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in Ws] if weights else []
    except Exception as ex:  # host memory too small for pinned copies
        return {"value": None, "unit": "TFLOP/s (algorithmic)", "error": str(ex)[:200]}
    for g, gh in zip(Gs, Gh):
        gh.copy_(g)
    torch.cuda.synchronize()
    groups = step_groups(shapes)
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    wp = [t.data_ptr() for t in Ws]
    gp = [t.data_ptr() for t in Gs]
    mp = [t.data_ptr() for t in Ms]

    def one_step():
        start = torch.cuda.Event()
        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)
        ready = []
        with torch.cuda.stream(h2d_s):
            for grp in groups:
                for i in grp:
                    Gs[i].copy_(Gh[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_s)
                ready.append(ev)
        for grp, ev in zip(groups, ready):
            stream.wait_event(ev)
            dm.dmuon_step_ptrs(h.h, [wp[i] for i in grp], [gp[i] for i in grp],
                               [mp[i] for i in grp], [shapes[i] for i in grp], 0.02, 0.95, 5,
                               stream=stream)
            if weights:
                done = torch.cuda.Event()
                done.record(stream)
                d2h_s.wait_event(done)
                with torch.cuda.stream(d2h_s):
                    for i in grp:
                        Wh[i].copy_(Ws[i], non_blocking=True)
        fin = torch.cuda.Event()
        fin.record(d2h_s)
        stream.wait_event(fin)
        if not weights:
            rc, _ = h.status(n_mats)   # the step's result: waits for it, reads its flags
            if rc != 0:
                raise RuntimeError("e2e status %d" % rc)

    one_step()  # plans the group shape list, fills the pointer-set cache
    torch.cuda.synchronize()
    h2d = sum(g.numel() * 4 for g in Gs)
    d2h = sum(x.numel() * 4 for x in Ws) if weights else 4 * (n_mats + 1)   # flags and the error word
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    rc, _ = h.status()
    if rc != 0:
        raise RuntimeError("e2e status %d" % rc)
    sec = e0.elapsed_time(e1) / 1e3
    del Gh, Wh
    return {"value": fl * args.e2e_steps * world / sec / 1e12, "unit": "TFLOP/s (algorithmic)",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": 1e3 * sec / args.e2e_steps, "groups": len(groups),
            "readback": "updated weights" if weights else "step status (dmuon_get_status)",
            "api": "dmuon_step per group, gradient uploads on a side stream"}


def free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def spawn_command(gpus, argv, port):
    """Command line that reruns this script as `gpus` ranks on this node
    (torchrun, rendezvous on 127.0.0.1), with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=%d" % gpus,
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def main():
    args = parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # --gpus N without a launcher: start the N ranks here (each replica
        # runs the whole workload; rank 0 prints the line)
        cmd = spawn_command(args.gpus, sys.argv[1:], free_port())
        os.execv(cmd[0], cmd)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit("bench.py: --gpus %d but WORLD_SIZE=%d" % (args.gpus, world))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
