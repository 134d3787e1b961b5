#!/usr/bin/env python3
"""Benchmark of the fused GMM EM step on GB300.

One step = one EM iteration over the whole workload (prepare, E-step with
log-sum-exp, statistics, reduction, M-step), inputs resident in HBM.
Prints ONE JSON line (rank 0).  Workloads are the synthetic ones of
datagen.WORKLOADS; the default is the largest one that fits one GPU: 2e8
points, D=128, K=1024, bf16 X (51 GB), diagonal EM, 5 iterations.

The timed steps are the workload's own EM schedule from theta_0 (its
iteration count unless --steps says otherwise), after --warmup untimed
iterations from theta_0; the value is the mean over the timed iterations,
and the line also gives each iteration's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--no-e2e]

--impl reference times the fp64 CPU oracle (the reference this path is
checked against) on a bounded sample of the same workload, on the host
cores.  Under torchrun (N > 1) each rank runs an independent replica of the
workload on its own GPU (the EM step is not sharded here): scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused EM step N*K pairs/s (1 x GB300)"
METRIC_ASSIGN = "top-m soft assignment N*K pairs/s (1 x GB300)"
UNIT = "pairs/s"
DEFAULT_WORKLOAD = "large_diag"
COV_NAMES = {0: "full", 1: "diag", 2: "iso"}
XNAMES = {0: "f32", 1: "f16", 2: "bf16"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                sm_max_mhz=2070.0, source="fallback")


# ---------------------------------------------------------------- work model

def slab_rows(wl):
    """Rows per screening launch of the tensor-core path (the library's rule)."""
    return 1 << 21


def tc_path(wl):
    """The tensor-core E-step runs for diagonal / isotropic covariance with
    D = 64 or 128 (the library's own rule)."""
    return wl.cov_type != 0 and wl.D in (64, 128)


def work_model(wl):
    """Algorithmic flops / bytes of one EM step and of each kernel (per launch).
    Diagonal / isotropic: the log-densities of all N*K pairs are the contraction
    [x, x^2] . [mu/var, -1/(2 var)], 2 * 2D flops per pair, plus 4D for the
    statistics; full: D(D+1) for the triangular solve and D(D+1) + 2D for the
    statistics.  The screening kernel is counted at one contraction of its
    rows (the EM mode runs exactly one; the assignment mode's streamed
    parameters two: bounds, then candidates); its bytes are its rows of X."""
    N, D, K = wl.N, wl.D, wl.K
    esz = 4 if wl.dtype == 0 else 2
    pairs = N * K
    if wl.cov_type == 0:
        e_flops, s_flops = D * (D + 1), D * (D + 1) + 2 * D
        pbytes = 4 * K * (1 + D + D * D)
    else:
        e_flops, s_flops = 4 * D, 4 * D
        pbytes = 4 * K * (1 + 2 * D)
    x_bytes = N * D * esz
    slabs = -(-N // slab_rows(wl))
    rows_per_launch = N / slabs
    return dict(
        pairs=pairs,
        step_flops=pairs * (e_flops + s_flops),
        step_bytes=x_bytes + 2 * pbytes,
        x_bytes=x_bytes,
        kernels={
            # tensor-core path: one screening launch per slab of rows
            "tc_screen_kernel": dict(flops=rows_per_launch * K * 4 * D,
                                     bytes=rows_per_launch * D * esz, bound="tensor",
                                     unit_note="%d-row slab" % round(rows_per_launch)),
            # CUDA-core path: the LSE pass computes every log-density; the
            # statistics pass recomputes them and accumulates the moments
            "lse_kernel": dict(flops=pairs * e_flops, bytes=x_bytes + 4 * N, bound="alu"),
            "stats_kernel": dict(flops=pairs * (e_flops + s_flops), bytes=x_bytes + 4 * N,
                                 bound="alu"),
            # full covariance, few components: the screen contracts every pair
            # (the triangular W_k x); the exact kernels take the candidate
            # pairs the status word counts (flops per pair below)
            "fc_screen_kernel": dict(flops=N * K * D * (D + 1), bytes=x_bytes, bound="tensor",
                                     unit_note="%d rows" % N),
            "fc_lse_kernel": dict(pair_flops=D * (D + 1), bound="alu"),
            "fc_stats_kernel": dict(pair_flops=2 * D * (D + 1) + 2 * D, bound="alu"),
            # streamed diagonal parameters: the dense-row kernels take the
            # candidate pairs of the rows the screen left them, the centred form
            # (x - mu)^2 w: 4 flops a dimension; the statistics recompute it and
            # add g y and g y^2: 4 more
            "dense_lse_kernel": dict(pair_flops=4 * D, bound="alu"),
            "dense_stats_kernel": dict(pair_flops=8 * D, bound="alu"),
        })


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception as e:  # no nvidia-smi
            log("clock sampling unavailable:", e)
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                                     hw=parts[5], hw_th=parts[6], sw_th=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                              ("sw_th", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in rows),
                    sm_max_mhz=max(r["sm_max"] for r in rows), samples=len(rows),
                    reasons=sorted(reasons))


# ---------------------------------------------------------------- helpers

def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu capture, if the kernel's
    sources are unchanged since it was taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload)
    if not rec:
        return None
    if rec.get("src_sha") != source_sha(rec.get("sources")):
        return None
    return rec.get("bytes_per_launch")


def source_sha(files=None):
    """Hash of the library sources `files` (names under csrc/; all of them
    when None): a capture stays valid while the kernel's own sources do."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "soft_clustering_gb300", "csrc")
    names = sorted(files) if files else sorted(
        fn for fn in os.listdir(csrc) if fn.endswith((".cu", ".cuh", ".h")))
    for fn in names:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, device=None):
    """The largest x over the ranks of the default process group (x itself
    without one): every rank's step time or end-to-end time, so the job's
    rate is set by its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput: the units every replica processed, over the
    slowest replica's time."""
    return world * units_per_rank / seconds


def oracle_params(wl, mix):
    """The parameters the oracle runs from: theta_0 and the EM options, or
    (assignment workloads) the planted parameters."""
    import datagen
    if wl.m:
        return datagen.planted_params_f16(mix), None
    theta = datagen.init_params(mix)
    return theta, datagen.em_opts(theta)


def oracle_once(wl, params, bits):
    """One oracle call on `bits`: an EM iteration from theta_0, or (assignment
    workloads) top-m against the planted parameters (`params` from
    oracle_params, made outside the timed call)."""
    import oracle
    (pi, mu, cov), opts = params
    if wl.m:
        return oracle.topm(bits, pi, mu, cov, wl.cov_type, wl.m, xdtype=wl.dtype)
    return oracle.em_step(bits, pi, mu, cov, wl.cov_type, xdtype=wl.dtype, opts=opts)


def cpu_sample_run(wl, mix, seconds):
    """The oracle (as it stands) on the first n' points of the workload, one
    EM iteration from theta_0; n' sized for about `seconds` of work.
    Returns (pairs_per_s, n', threads, seconds_taken)."""
    import datagen
    import oracle
    params = oracle_params(wl, mix)
    # calibrate on growing samples until one takes a second or more: small
    # samples leave most threads idle (the oracle parallelises over blocks
    # of points), so their time per point overstates a large sample's
    n_cal = min(wl.N, 16384)
    while True:
        bits = datagen.points(mix, 0, n_cal)
        t0 = time.perf_counter()
        oracle_once(wl, params, bits)
        dt = time.perf_counter() - t0
        per_point = max(dt / n_cal, 1e-9)
        if dt >= 1.0 or n_cal >= wl.N:
            break
        n_cal = int(min(wl.N, max(2 * n_cal, 1.5 / per_point)))
    n = int(min(wl.N, max(n_cal, seconds / per_point)))
    bits = datagen.points(mix, 0, n)
    t0 = time.perf_counter()
    oracle_once(wl, params, bits)
    dt = time.perf_counter() - t0
    return n * wl.K / dt, n, oracle.max_threads(), dt


# ---------------------------------------------------------------- arms

def run_reference(args, wl):
    """The fp64 oracle timed on the host cores on a bounded sample per step."""
    import datagen
    import oracle
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    mix = datagen.planted(wl)
    total_steps = args.steps + args.warmup
    per_step_s = max(2.0, min(20.0, 150.0 / max(total_steps, 1)))
    _, n, threads, _ = cpu_sample_run(wl, mix, per_step_s)
    bits = datagen.points(mix, 0, n)
    times = []
    if wl.m:
        pi, mu, var = datagen.planted_params_f16(mix)
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.topm(bits, pi, mu, var, wl.cov_type, wl.m, xdtype=wl.dtype)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        what = "one top-%d assignment per step" % wl.m
    else:
        theta = datagen.init_params(mix)
        opts = datagen.em_opts(theta)
        pi, mu, cov = theta
        for _ in range(args.warmup):
            r = oracle.em_step(bits, pi, mu, cov, wl.cov_type, xdtype=wl.dtype, opts=opts)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            r = oracle.em_step(bits, pi, mu, cov, wl.cov_type, xdtype=wl.dtype, opts=opts)
            times.append(time.perf_counter() - t0)
            pi, mu, cov = r["pi"], r["mu"], r["cov"]
        what = "one EM iteration per step"
    ms = 1e3 * sum(times) / len(times)
    value = n * wl.K / (ms / 1e3)
    sample = "first %d of %d points, %s (fp64 oracle)" % (n, wl.N, what)
    line = dict(metric=METRIC_ASSIGN if wl.m else METRIC, value=value, unit=UNIT, n_gpus=world,
                steps=args.steps,
                warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=config_dict(wl, extra=dict(sample_points=n)),
                cpu_baseline=dict(value=value, unit=UNIT, cores=threads, kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def config_dict(wl, extra=None):
    d = dict(workload=wl.name, N=wl.N, D=wl.D, K=wl.K, cov=COV_NAMES[wl.cov_type],
             x_dtype=XNAMES[wl.dtype], l2="inputs larger than L2 (X is %.2f GB > 129 MB)"
             % (wl.N * wl.D * (4 if wl.dtype == 0 else 2) / 1e9))
    if extra:
        d.update(extra)
    return d


def run_ours(args, wl):
    import numpy as np
    import torch
    import datagen
    import soft_clustering_gb300 as G
    from soft_clustering_gb300 import build as gbuild
    from soft_clustering_gb300.torch_api import GMMState

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        gbuild.build()
    if world > 1:
        torch.distributed.barrier()
    G.lib()
    peaks = measured_peaks()
    wm = work_model(wl)

    # inputs: drawn straight into HBM (same bits the host generator gives)
    mix = datagen.planted(wl)
    keep, ptrs = datagen.upload_tables(mix, device=dev)
    esz = 4 if wl.dtype == 0 else 2
    X = torch.empty(wl.N * wl.D * esz, dtype=torch.uint8, device=dev)
    datagen.device_points(mix, 0, wl.N, X.data_ptr(), torch.cuda.current_stream().cuda_stream,
                          ptrs)
    theta0 = datagen.init_params(mix)
    torch.cuda.synchronize()

    opts = datagen.em_opts(theta0)
    st = GMMState(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, device=dev)
    for k, v in opts.items():
        setattr(st.opts, k, v)
    steps = args.steps
    # warm-up: W untimed iterations from theta_0
    st.set_params(*theta0)
    for _ in range(args.warmup):
        st.step(X)
    torch.cuda.synchronize()
    status = st.device_status()
    if status != 0:
        log("device status after warm-up:", G.status_string(status))

    # timed region: the workload's EM schedule from theta_0 on device-resident
    # X, CUDA events on the launching stream (one per iteration)
    st.set_params(*theta0)
    G.gmm_profile_reset()
    G.gmm_profile_enable(True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(steps):
        st.step(X)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    G.gmm_profile_enable(False)
    prof = G.gmm_profile_read()
    per_iter = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    ms = max_over_ranks(evs[0].elapsed_time(evs[-1]) / steps, dev)
    status = st.device_status()
    ll = float(st.loglik.item())
    value = job_rate(world, wm["pairs"], ms / 1e3)
    launches = sum(n for (_, n) in prof.values())

    # dominant kernel roofline, measured live in the timed region
    top = max(prof.items(), key=lambda kv: kv[1][0])[0] if prof else None
    roof = None
    if top:
        tot_ms, n_launch = prof[top]
        avg_s = tot_ms / n_launch / 1e3
        km = wm["kernels"].get(top)
        if km and "pair_flops" in km:
            # candidate-driven kernel: replay the timed schedule (untimed, from
            # theta_0) and count the pairs it evaluated from the status word
            st.set_params(*theta0)
            cand_pairs = 0
            for _ in range(steps):
                st.step(X)
                cand_pairs += int(st.ws[16:24].cpu().numpy().view(np.uint64)[0])
            km = dict(km, flops=cand_pairs * km["pair_flops"] / n_launch,
                      pairs_per_launch=cand_pairs / n_launch)
        if km and km["bound"] == "tensor":
            # fp16 operands, fp32 accumulation: the dense fp16 rate equals the
            # bf16 rate (nominal ratio 1), so the measured bf16 GEMM peak is used
            peak = peaks["bf16_tflops"]
            achieved = km["flops"] / avg_s / 1e12
            roof = dict(bound="tensor", achieved=achieved, peak=peak, unit="TFLOP/s",
                        frac=achieved / peak, traffic=traffic_for(top, wl.name),
                        kernel=top, avg_launch_ms=tot_ms / n_launch,
                        per_launch=km["unit_note"],
                        hbm_achieved_gbs=km["bytes"] / avg_s / 1e9,
                        peak_source="bf16 dense GEMM, %s (fp16 = bf16 rate)" % peaks["source"])
        elif km:
            # CUDA-core fp32 kernels: ALU peak = 152 SMs x 128 lanes x 2 flops x max SM clock
            alu_peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            achieved = km["flops"] / avg_s / 1e12
            roof = dict(bound="alu", achieved=achieved, peak=alu_peak, unit="TFLOP/s",
                        frac=achieved / alu_peak, traffic=traffic_for(top, wl.name),
                        kernel=top, avg_launch_ms=tot_ms / n_launch,
                        peak_source="fp32 FMA lanes x clock (derived)")
            if "pairs_per_launch" in km:
                roof["per_launch"] = "%.4g candidate pairs x %d flops" % (
                    km["pairs_per_launch"], km["pair_flops"])
    step_roof_s = max(wm["step_flops"] / (peaks["bf16_tflops"] * 1e12),
                      wm["step_bytes"] / (peaks["hbm_gbs"] * 1e9))

    # end to end through the host-buffer entry point: X streamed from pinned
    # host memory every iteration, the log-likelihood read back every
    # iteration; the same schedule (W untimed iterations from theta_0, then
    # the timed ones from theta_0)
    e2e = None
    if not args.no_e2e:
        chunk = max(1, min(wl.N, (256 << 20) // (wl.D * esz)))
        st2 = GMMState(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, device=dev, chunk_rows=chunk)
        for k, v in opts.items():
            setattr(st2.opts, k, v)
        host = torch.empty(wl.N * wl.D * esz, dtype=torch.uint8, pin_memory=True)
        host.copy_(X)
        ll_host = torch.zeros(1, dtype=torch.float64, pin_memory=True)
        del X
        del st
        torch.cuda.empty_cache()
        st2.set_params(*theta0)
        for _ in range(args.warmup):
            st2.step_host(host, loglik_host=ll_host)
        st2.set_params(*theta0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            st2.step_host(host, loglik_host=ll_host)
        e2e_s = max_over_ranks((time.perf_counter() - t0) / steps, dev)
        e2e = dict(value=job_rate(world, wm["pairs"], e2e_s), unit=UNIT,
                   h2d_bytes_per_step=wm["x_bytes"], d2h_bytes_per_step=8,
                   ms_per_step=e2e_s * 1e3, chunk_rows=chunk)
        del host

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, thr, dt = cpu_sample_run(wl, mix, 12.0)
        cpu = dict(value=v, unit=UNIT, cores=thr, kind="oracle",
                   sample="first %d of %d points, one EM iteration from theta_0, %.1f s" %
                   (n, wl.N, dt))

    if rank == 0:
        line = dict(
            metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
            vs_baseline=None, dtype="f32", data="synthetic",
            # f32: exact log-densities, log-sum-exp and statistics; the
            # screening contraction runs on fp16 tensor cores (fp32 accumulate)
            config=config_dict(wl, extra=dict(
                iters_per_s=1e3 / ms, parallelism="replicas" if world > 1 else "single",
                schedule="iterations 0..%d from theta_0 (after %d untimed ones from theta_0)"
                         % (steps - 1, args.warmup),
                ms_per_iteration=[round(t, 4) for t in per_iter],
                steady_ms_per_step=per_iter[-1],
                e_step="tensor-core screen (fp16) + exact fp32 refine" if tc_path(wl)
                else "CUDA-core fp32",
                loglik=ll, device_status=G.status_string(status),
                step_roofline=dict(flops=wm["step_flops"], bytes=wm["step_bytes"],
                                   roofline_ms=step_roof_s * 1e3,
                                   frac=step_roof_s * 1e3 / ms,
                                   peaks="bf16 %.1f TFLOP/s, HBM %.1f GB/s (%s)" % (
                                       peaks["bf16_tflops"], peaks["hbm_gbs"], peaks["source"])),
                kernels={k: dict(ms_per_launch=v[0] / v[1], launches=v[1])
                         for k, v in prof.items()})),
            roofline=roof, cpu_baseline=cpu, e2e=e2e, gpu_launches=launches, clocks=clk)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_assign(args, wl):
    """Top-m soft assignment of every point against the planted parameters
    (the IVF multi-assignment workload): gmm_assign_topm on device-resident X;
    e2e copies X in from pinned host memory and the ids / gamma out, every step."""
    import torch
    import datagen
    import soft_clustering_gb300 as G
    from soft_clustering_gb300 import build as gbuild
    from soft_clustering_gb300.torch_api import Assigner

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        gbuild.build()
    if world > 1:
        torch.distributed.barrier()
    G.lib()
    peaks = measured_peaks()
    wm = work_model(wl)
    mix = datagen.planted(wl)
    keep, ptrs = datagen.upload_tables(mix, device=dev)
    esz = 4 if wl.dtype == 0 else 2
    X = torch.empty(wl.N * wl.D * esz, dtype=torch.uint8, device=dev)
    datagen.device_points(mix, 0, wl.N, X.data_ptr(), torch.cuda.current_stream().cuda_stream,
                          ptrs)
    pi, mu, var = datagen.planted_params_f16(mix)
    a = Assigner(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, wl.m, device=dev)
    a.prepare(pi, mu, var)
    for _ in range(args.warmup):
        a.assign(X)
    torch.cuda.synchronize()
    status = a.device_status()
    if status != 0:
        log("device status after warm-up:", G.status_string(status))

    G.gmm_profile_reset()
    G.gmm_profile_enable(True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        a.assign(X)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    G.gmm_profile_enable(False)
    prof = G.gmm_profile_read()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dev)
    status = a.device_status()
    value = job_rate(world, wm["pairs"], ms / 1e3)
    launches = sum(n for (_, n) in prof.values())
    top = max(prof.items(), key=lambda kv: kv[1][0])[0] if prof else None
    roof = None
    if top and top in wm["kernels"] and wm["kernels"][top]["bound"] == "tensor":
        km = wm["kernels"][top]
        tot_ms, n_launch = prof[top]
        avg_s = tot_ms / n_launch / 1e3
        achieved = km["flops"] / avg_s / 1e12
        roof = dict(bound="tensor", achieved=achieved, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=achieved / peaks["bf16_tflops"], traffic=traffic_for(top, wl.name),
                    kernel=top, avg_launch_ms=tot_ms / n_launch, per_launch=km["unit_note"],
                    hbm_achieved_gbs=km["bytes"] / avg_s / 1e9,
                    peak_source="bf16 dense GEMM, %s (fp16 = bf16 rate)" % peaks["source"])
    # assignment roofline: 4NKD flops (no statistics), one read of X + the outputs
    out_bytes = wl.N * wl.m * 8 + wl.N * 4
    step_roof_s = max(wl.N * wl.K * 4 * wl.D / (peaks["bf16_tflops"] * 1e12),
                      (wm["x_bytes"] + out_bytes) / (peaks["hbm_gbs"] * 1e9))

    e2e = None
    if not args.no_e2e:
        host = torch.empty(wl.N * wl.D * esz, dtype=torch.uint8, pin_memory=True)
        host.copy_(X)
        ids_h = torch.empty(wl.N, wl.m, dtype=torch.int32, pin_memory=True)
        gam_h = torch.empty(wl.N, wl.m, dtype=torch.float32, pin_memory=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            X.copy_(host, non_blocking=True)
            a.assign(X, with_lse=False)
            ids_h.copy_(a.ids, non_blocking=True)
            gam_h.copy_(a.gamma, non_blocking=True)
            torch.cuda.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, dev)
        e2e = dict(value=job_rate(world, wm["pairs"], e2e_s), unit=UNIT, h2d_bytes_per_step=wm["x_bytes"],
                   d2h_bytes_per_step=wl.N * wl.m * 8, ms_per_step=e2e_s * 1e3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, thr, dt = cpu_sample_run(wl, mix, 12.0)
        cpu = dict(value=v, unit=UNIT, cores=thr, kind="oracle",
                   sample="first %d of %d points, top-%d assignment, %.1f s" % (n, wl.N, wl.m, dt))
    if rank == 0:
        line = dict(
            metric=METRIC_ASSIGN, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
            vs_baseline=None, dtype="f32", data="synthetic",
            config=config_dict(wl, extra=dict(
                m=wl.m, parallelism="replicas" if world > 1 else "single",
                device_status=G.status_string(status),
                step_roofline=dict(flops=wl.N * wl.K * 4 * wl.D,
                                   bytes=wm["x_bytes"] + out_bytes,
                                   roofline_ms=step_roof_s * 1e3, frac=step_roof_s * 1e3 / ms),
                kernels={k: dict(ms_per_launch=v[0] / v[1], launches=v[1])
                         for k, v in prof.items()})),
            roofline=roof, cpu_baseline=cpu, e2e=e2e, gpu_launches=launches, clocks=clk)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed iterations (default: the workload's own EM schedule; 5 for "
                         "assignment workloads)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--n", type=int, default=None,
                    help="override the number of points (small profiling cases)")
    args = ap.parse_args(argv)
    import datagen
    wl = datagen.WORKLOADS[args.workload]
    if args.n:
        wl = wl.with_n(args.n)
    if args.steps is None:
        args.steps = wl.iters if not wl.m else 5
    if args.impl == "reference":
        return run_reference(args, wl)
    if wl.m:
        return run_assign(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
