"""Benchmark of the selective-scan forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one full pass of the hot path (one call of the operation) over the
workload's synthetic inputs, already resident in HBM.  The default workload
is the Vim-S 1248x1248 bidirectional v2 scan: batch 8, d_inner 768,
d_state 16, L = 78*78 + 1 = 6085, bf16 I/O with fp32 state.

One JSON line is printed by rank 0.  `value` is the algorithmic HBM
throughput (every I/O tensor read once, y written once) of the whole job in
GB/s; `elem_updates_per_s` counts (direction, batch, channel, state, step)
recurrence updates.  Inputs are larger than L2, so no flush is needed between
steps.  Under torchrun every rank runs its own replica with its own seed
(rows are independent: weak scaling, no collective on the data path).

`--impl reference` times the fp64 CPU oracle (the reference of this
repository) on a bounded sample of whole rows of the same workload, on the
host cores, and prints the same metric.
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

DEFAULT_WORKLOAD = "vim_s_1248_bimamba_v2"
METRIC = "bi-dir selective-scan HBM GB/s (% of peak) and elem-updates/s, Vim-S 1248²"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2032.0)), "measured"
    return 6400.0, 2032.0, "fallback"


def bf16_peak_tflops():
    """Dense bf16 tensor peak for a kernel timed on its own (burst)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    return 1800.0, "fallback"


# ---------------------------------------------------------------- GPU arm
def launches_per_step(op):
    """Kernels one call launches: B/C packing (one launch for every B/C
    set), the transposes of SS2D, and the scan kernel(s)."""
    return {"single": 2, "v1": 2, "v2": 2, "ss2d": 5}[op]


def scan_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("bidir_kernel.cuh", "scan_ops.cuh"):
        with open(os.path.join(ROOT, "selective_state_space_111_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    """DRAM bytes per launch of the scan kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "scan_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    ent = d.get(workload)
    if not ent or ent.get("src_sha") != scan_sources_sha():
        return None
    return ent.get("dram_bytes_per_launch")


def alu_rates():
    """Lane operations per SM per clock of scalar FMA, packed FMA and MUFU
    2^x on this GPU (the microbenchmark in csrc/alu_rates.cu), or None."""
    import ctypes
    try:
        from selective_state_space_111_b300 import build
        lib = ctypes.CDLL(build.build_alu())
        out = (ctypes.c_double * 3)()
        if lib.ssm_alu_rates(out) != 0:
            return None
    except (OSError, subprocess.CalledProcessError):
        return None
    r = {"ffma": round(out[0], 1), "ffma2": round(out[1], 1), "mufu_ex2": round(out[2], 1)}
    # element updates per SM per clock each pipe allows: 4 FMA-pipe operations
    # and one MUFU ex2 per update
    r["updates_per_sm_clock"] = round(min(max(out[0], out[1]) / 4, out[2]), 2)
    return r


# ---------------------------------------------------------------- ranks
def rank_env():
    """(world, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(workload, rank):
    """Each replica draws its own inputs: the workload's seed plus the rank."""
    from selective_state_space_111_b300.synth import seed_for
    return seed_for(workload) + rank


def max_over_ranks(value, world, device=None):
    """The slowest rank's time (the job's time): an all-reduce MAX of one
    float (a no-op alone).  Replicas share nothing else."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def call(ssm, spec, g, ws, out):
    sp = spec.delta_softplus
    if spec.op == "single":
        return ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                      g["delta_bias"], sp, out=out, workspace=ws)
    if spec.op == "v1":
        return ssm.bimamba_scan_fwd_v1(g["u"], g["delta"], g["A"], g["A_b"], g["B"], g["C"],
                                       g["D"], g["z"], g["delta_bias"], sp, g["out_scale"],
                                       out=out, workspace=ws)
    if spec.op == "v2":
        return ssm.bimamba_scan_fwd_v2(g["u"], g["delta"], g["delta_b"], g["A"], g["A_b"], g["B"],
                                       g["C"], g["B_b"], g["C_b"], g["D"], g["D_b"], g["z"],
                                       g["delta_bias"], g["delta_bias_b"], g["u_b"], sp,
                                       g["out_scale"], out=out, workspace=ws)
    return ssm.ss2d_scan_fwd(g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                             g["delta_bias"], sp, out=out, workspace=ws)


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        # "under load": samples at the upper half of the observed power range
        if pw:
            thr = min(pw) + 0.5 * (max(pw) - min(pw))
            loaded = [num(r[1]) for r in rows if num(r[3]) is not None and num(r[3]) >= thr
                      and num(r[1]) is not None]
        else:
            loaded = sm
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from selective_state_space_111_b300 import build
    build.build()
    import selective_state_space_111_b300 as ssm
    from selective_state_space_111_b300.synth import WORKLOADS, make_inputs

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    spec = WORKLOADS[args.workload]
    t = make_inputs(spec, rank_seed(args.workload, rank))
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    L = spec.seq_len
    ws_n = ssm.workspace_bytes(spec.op, g["u" if spec.op != "ss2d" else "x"].dtype, spec.B,
                               spec.D, L, spec.N, spec.K)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)
    out = torch.empty_like(g["x"] if spec.op == "ss2d" else g["u"])
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        call(ssm, spec, g, ws, out)
    torch.cuda.synchronize()

    # The timed region: windows of exactly K steps, each bracketed by a
    # barrier and a synchronize on both sides, repeated until the windows
    # add up to at least --min-seconds of device time, with the SM clock and
    # throttle reasons sampled throughout.  ms_per_step is the median
    # window's; the scan kernel's own time comes from the library's
    # profiling hook around each of its launches.
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    for e in kb + ke:
        e.record(stream)                  # creates the CUDA events
    torch.cuda.synchronize()

    def window():
        barrier()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(args.steps):
            ssm.set_profile_events(kb[i], ke[i])
            call(ssm, spec, g, ws, out)
            ev[i + 1].record(stream)
        ssm.set_profile_events(None, None)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[-1]), [kb[i].elapsed_time(ke[i]) for i in range(args.steps)]

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)                      # the sampler's first reading
    wins, kern = [], []
    spent = 0.0
    while not wins or (spent < args.min_seconds * 1e3 and len(wins) < 10000):
        w_ms, k_ms = window()
        wins.append(w_ms)
        kern.extend(k_ms)
        spent += w_ms
    clocks = sampler.stop()
    total_ms = statistics.median(wins)
    total_ms = max_over_ranks(total_ms, world, dev)

    # e2e: host (pinned) inputs -> device -> the public API -> result to host,
    # every step.  Steps are pipelined the way a serving loop runs them: the
    # upload of step k+1 (copy stream) and the download of step k-1 (second
    # copy stream) overlap the scan of step k, with two device buffer sets.
    e2e = None
    if not args.no_e2e:
        host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
        d2h = h_out.numel() * h_out.element_size()
        n_e2e = max(1, min(args.steps, 20))
        nb = 2
        bufs = [{k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else v)
                 for k, v in host.items()} for _ in range(nb)]
        outs = [torch.empty_like(out) for _ in range(nb)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_comp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]

        def e2e_step(k):
            i = k % nb
            with torch.cuda.stream(s_in):
                if k >= nb:
                    s_in.wait_event(ev_comp[i])         # buffer set i is free again
                for name, v in host.items():
                    if isinstance(v, torch.Tensor):
                        bufs[i][name].copy_(v, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if k >= nb:
                stream.wait_event(ev_out[i])            # out buffer i downloaded
            call(ssm, spec, bufs[i], ws, outs[i])
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                h_out.copy_(outs[i], non_blocking=True)
                ev_out[i].record(s_out)

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for k in range(n_e2e):
            e2e_step(k)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": round(spec.algorithmic_bytes() * world / (e2e_ms * 1e-3) / 1e9, 3),
               "unit": "GB/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_ms, 4), "pipelined": "upload k+1 / scan k / download k-1"}
        if not torch.equal(h_out.to(dev), outs[(n_e2e - 1) % nb]):
            raise RuntimeError("e2e: downloaded result differs from the device result")

    # NVTX ranges name the backward and prologue legs, so a profiler can
    # select their launches (ncu --nvtx --nvtx-include "backward/")
    bwd = None
    if not args.no_backward:
        bwd = measure_backward(ssm, spec, g, t, dev, stream, max(3, min(args.steps, 20)))
    pro = None
    if not args.no_prologue:
        torch.cuda.nvtx.range_push("prologue")
        pro = measure_prologue(ssm, spec, dev, stream, max(3, min(args.steps, 20)))
        torch.cuda.nvtx.range_pop()
    opj = None
    if not args.no_out_proj:
        torch.cuda.nvtx.range_push("out_proj")
        opj = measure_out_proj(ssm, spec, dev, stream, max(3, min(args.steps, 20)))
        torch.cuda.nvtx.range_pop()

    if rank == 0:
        ms = total_ms / args.steps
        hbm_peak, sm_max, peak_kind = peaks()
        gbps = spec.algorithmic_bytes() * world / (ms * 1e-3) / 1e9
        ups = spec.updates() * world / (ms * 1e-3)
        # dominant kernel: the scan kernel's average launch over the timed region
        kern_ms = statistics.mean(kern)
        scans = 2 if spec.op == "ss2d" else 1          # the hook brackets the last one
        upd_launch = spec.updates() / scans
        # ALU roof: 128 fp32 lanes per SM and 4 fp32 operations per element
        # update (equal to the MUFU ex2 roof: 32 per SM per clock, one each)
        alu_peak = 148 * 32 * sm_max * 1e6 / 1e9          # Gupd/s
        alu_ach = upd_launch / (kern_ms * 1e-3) / 1e9
        sm_run = clocks.get("sm_mhz") or sm_max           # the clock the kernel ran at
        alu_peak_run = 148 * 32 * sm_run * 1e6 / 1e9
        rates = alu_rates()
        line = {
            "metric": METRIC,
            "value": round(gbps, 2),
            "unit": "GB/s",
            "pct_of_hbm_peak": round(100 * gbps / hbm_peak, 2),
            "elem_updates_per_s": float("%.4g" % ups),
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 5),
            "timed_windows": {"windows": len(wins), "steps_each": args.steps,
                              "device_s": round(spent / 1e3, 3),
                              "ms_per_step_min": round(min(wins) / args.steps, 5),
                              "ms_per_step_max": round(max(wins) / args.steps, 5)},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if spec.io == "bf16" else "f32",
            "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
            "config": {"workload": args.workload, "op": spec.op, "batch": spec.B,
                       "d_inner": spec.D, "d_state": spec.N, "seq_len": L,
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "alu", "achieved": round(alu_ach, 2), "peak": round(alu_peak, 1),
                         "unit": "Gupd/s", "frac": round(alu_ach / alu_peak, 4),
                         "traffic": (args.traffic if args.traffic is not None
                                     else measured_traffic(args.workload)),
                         "kernel": "bidir_scan_kernel", "kernel_ms": round(kern_ms, 5),
                         "peak_basis": "148 SMs x 128 fp32 lanes x %.0f MHz / 4 fp32 ops per "
                                       "update (recipe unit counts and max clock)" % sm_max,
                         "frac_at_sampled_clock": round(alu_ach / alu_peak_run, 4),
                         "sampled_sm_mhz": sm_run,
                         "alu_rates_per_sm_clock": rates,
                         "hbm_gbs_kernel": round(spec.algorithmic_bytes() / scans
                                                 / (kern_ms * 1e-3) / 1e9, 1),
                         "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": peak_kind},
            "gpu_launches": launches_per_step(spec.op) * args.steps,
            "clocks": clocks,
        }
        if e2e:
            line["e2e"] = e2e
        if bwd:
            # ALU roof of the backward: 16 fp32 operations per element update
            # (3 to recompute the state, 13 for the adjoint step)
            bpeak = 148 * 128 * sm_max * 1e6 / 16 / 1e9
            bach = spec.updates() / (bwd["ms"] * 1e-3) / 1e9
            bwd["value"] = round(spec.backward_bytes() / (bwd["ms"] * 1e-3) / 1e9, 2)
            bwd["unit"] = "GB/s"
            bwd["roofline"] = {"bound": "alu", "achieved": round(bach, 2),
                               "peak": round(bpeak, 1), "unit": "Gupd/s",
                               "frac": round(bach / bpeak, 4),
                               "peak_basis": "148 SMs x 128 fp32 lanes x %.0f MHz / 16 fp32 "
                                             "ops per update" % sm_max}
            fc = bwd.get("from_context")
            if fc:
                cach = spec.updates() / (fc["ms"] * 1e-3) / 1e9
                fc["roofline"] = {"bound": "alu", "achieved": round(cach, 2),
                                  "peak": round(bpeak, 1), "unit": "Gupd/s",
                                  "frac": round(cach / bpeak, 4)}
                del fc["ms"]
            line["backward"] = bwd
        if pro:
            # the projections are skinny (x_proj d_inner -> dt_rank + 2 d_state,
            # dt_proj dt_rank -> d_inner): the prologue is bound by moving x, u
            # and the projections' outputs, so its roof is HBM bandwidth over
            # its algorithmic bytes; the contraction rate is reported beside it
            pro["roofline"] = {"bound": "hbm", "achieved": pro["value"], "peak": hbm_peak,
                               "unit": "GB/s", "frac": round(pro["value"] / hbm_peak, 4),
                               "peak_kind": peak_kind,
                               "tflops": round(pro.pop("tflops"), 3)}
            line["prologue"] = pro
        if opj:
            # a dense contraction (d_inner -> d_model per position): its roof
            # is the tensor peak of its dtype (fp16 at bf16's rate); the
            # HBM fraction of its bytes is reported beside it
            tpk, tkind = bf16_peak_tflops()
            opj["roofline"] = {"bound": "tensor", "achieved": opj["tflops"], "peak": tpk,
                               "unit": "TFLOP/s", "frac": round(opj["tflops"] / tpk, 4),
                               "peak_kind": tkind,
                               "hbm_frac": round(opj["value"] / hbm_peak, 4)}
            line["out_proj"] = opj
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(spec, args.workload, args.cpu_seconds)
            line["cpu_baseline_single_thread"] = cpu_baseline(spec, args.workload,
                                                              args.cpu_seconds / 2, threads=1)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_backward(ssm, spec, g, t, dev, stream, steps):
    """Time the backward call (gradients of sum(dout * out)) on the same
    inputs: 3 warm-up calls, then `steps` calls between CUDA events."""
    import torch
    gen = torch.Generator().manual_seed(12345)
    shape = t["x" if spec.op == "ss2d" else "u"].shape
    dout = torch.randn(shape, generator=gen).to(dtype=g["x" if spec.op == "ss2d" else "u"].dtype,
                                                device=dev)
    L = spec.seq_len
    ws = torch.empty(max(1, ssm.bwd_workspace_bytes(spec.op, dout.dtype, spec.B, spec.D, L,
                                                    spec.N, spec.K,
                                                    spec.op == "v2" and not spec.shared_u)),
                     dtype=torch.uint8, device=dev)
    sp = spec.delta_softplus

    def once():
        if spec.op == "single":
            return ssm.selective_scan_bwd(dout, g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"],
                                          g["z"], g["delta_bias"], sp, workspace=ws)
        if spec.op == "v1":
            return ssm.bimamba_scan_bwd_v1(dout, g["u"], g["delta"], g["A"], g["A_b"], g["B"],
                                           g["C"], g["D"], g["z"], g["delta_bias"], sp,
                                           g["out_scale"], workspace=ws)
        if spec.op == "v2":
            return ssm.bimamba_scan_bwd_v2(dout, g["u"], g["delta"], g["delta_b"], g["A"],
                                           g["A_b"], g["B"], g["C"], g["B_b"], g["C_b"], g["D"],
                                           g["D_b"], g["z"], g["delta_bias"], g["delta_bias_b"],
                                           g["u_b"], sp, g["out_scale"], workspace=ws)
        return ssm.ss2d_scan_bwd(dout, g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                 g["delta_bias"], sp, workspace=ws)

    torch.cuda.nvtx.range_push("backward")
    for _ in range(3):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        once()
    e1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms = e0.elapsed_time(e1) / steps
    res = {"ms_per_call": round(ms, 4), "ms": ms, "steps": steps,
           "bytes_per_call": spec.backward_bytes(),
           "elem_updates_per_s": float("%.4g" % (spec.updates() / (ms * 1e-3)))}
    if spec.op in ("single", "v1", "v2") and spec.N <= 16:
        # the training pairing: the forward call leaves the backward's context
        # (pre-gate output, chunk-start states) and the backward call reads it
        # instead of running the forward pass again; both timed (in an NVTX
        # range of their own)
        torch.cuda.nvtx.range_push("backward_from_context")
        n = ssm.bwd_context_bytes(spec.op, dout.dtype, spec.B, spec.D, L, spec.N)
        ctx = torch.empty(n, dtype=torch.uint8, device=dev)
        fws = torch.empty(max(16, ssm.workspace_bytes(spec.op, dout.dtype, spec.B, spec.D, L,
                                                      spec.N, spec.K)),
                          dtype=torch.uint8, device=dev)
        out = torch.empty_like(dout)
        ssm.set_bwd_context(ctx)
        try:
            for _ in range(3):
                call(ssm, spec, g, fws, out)
                once()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(steps):
                call(ssm, spec, g, fws, out)
            e1.record(stream)
            torch.cuda.synchronize()
            f_ms = e0.elapsed_time(e1) / steps
            e0.record(stream)
            for _ in range(steps):
                once()
            e1.record(stream)
            torch.cuda.synchronize()
            b_ms = e0.elapsed_time(e1) / steps
        finally:
            ssm.set_bwd_context(None)
            torch.cuda.nvtx.range_pop()
        res["from_context"] = {"ms_per_call": round(b_ms, 4), "ms": b_ms,
                               "forward_ms_per_call": round(f_ms, 4), "context_bytes": n}
    return res


def measure_out_proj(ssm, spec, dev, stream, steps):
    """Time the block's output projection (d_inner -> d_model = d_inner / 2,
    the pages' ssm_ratio / expand of 2) on a gated output of the workload's
    shape: out = W_out y, synthetic weights in the I/O dtype."""
    import torch
    B, D, L = spec.B, spec.D, spec.seq_len
    Dm = D // 2
    gen = torch.Generator().manual_seed(2468)
    io = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[spec.io]
    y = torch.randn(B, D, L, generator=gen).to(dtype=io, device=dev)
    W = (torch.randn(Dm, D, generator=gen) * D ** -0.5).to(dtype=io, device=dev)
    for _ in range(3):
        ssm.out_proj_fwd(y, W)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        ssm.out_proj_fwd(y, W)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    e = y.element_size()
    nbytes = e * (B * D * L + Dm * D + B * Dm * L)        # y and W read, out written
    flops = 2.0 * B * L * D * Dm
    return {"ms_per_call": round(ms, 4), "d_inner": D, "d_model": Dm,
            "value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2)}


def measure_prologue(ssm, spec, dev, stream, steps):
    """Time the prologue that feeds the scan (conv1d + SiLU, x_proj, dt_proj)
    on an input of the workload's shape: both branches for v2 (the backward
    one on the flipped input), one for v1 (shared weights) and single; for
    SS2D the 3x3 conv2d + SiLU and the four directions' projections.
    dt_rank = ceil(d_model / 16) with d_model = D / 2; weights synthetic."""
    import torch
    B, D, L, N = spec.B, spec.D, spec.seq_len, spec.N
    R, K = -(-D // 32), 4
    if spec.op == "ss2d":
        return measure_ss2d_prologue(ssm, spec, dev, stream, steps, R)
    dirs = 2 if spec.op == "v2" else 1
    gen = torch.Generator().manual_seed(4321)
    io = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[spec.io]
    x = torch.randn(B, D, L, generator=gen).to(dtype=io, device=dev)
    w = [dict(conv_w=(torch.rand(D, K, generator=gen) - 0.5).to(dev),
              conv_b=(torch.rand(D, generator=gen) - 0.5).to(dev),
              W_x=(torch.randn(R + 2 * N, D, generator=gen) * D ** -0.5).to(dev),
              W_dt=(torch.randn(D, R, generator=gen) * R ** -0.5).to(dev)) for _ in range(dirs)]
    ws = torch.empty(B * R * L * 4, dtype=torch.uint8, device=dev)

    def once():
        for k in range(dirs):
            ssm.mamba_prologue_fwd(x, w[k]["conv_w"], w[k]["conv_b"], w[k]["W_x"], w[k]["W_dt"],
                                   R, N, reverse=k == 1, workspace=ws)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        once()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    e = x.element_size()
    # per direction: x read; u, dt written [B,D,L]; B, C written [B,N,L]
    nbytes = dirs * e * (3 * B * D * L + 2 * B * N * L)
    flops = dirs * 2.0 * B * L * ((R + 2 * N) * D + D * R)
    return {"ms_per_call": round(ms, 4), "directions": dirs, "dt_rank": R, "d_conv": K,
            "value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "tflops": flops / (ms * 1e-3) / 1e12}


def measure_ss2d_prologue(ssm, spec, dev, stream, steps, R, Kc=3):
    import torch
    B, D, H, W, N = spec.B, spec.D, spec.H, spec.W, spec.N
    L = H * W
    gen = torch.Generator().manual_seed(4322)
    io = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[spec.io]
    x = torch.randn(B, D, H, W, generator=gen).to(dtype=io, device=dev)
    w = dict(conv_w=((torch.rand(D, Kc, Kc, generator=gen) - 0.5) / Kc).to(dev),
             conv_b=(torch.rand(D, generator=gen) - 0.5).to(dev),
             W_x=(torch.randn(4, R + 2 * N, D, generator=gen) * D ** -0.5).to(dev),
             W_dt=(torch.randn(4, D, R, generator=gen) * R ** -0.5).to(dev))
    ws = torch.empty(B * 4 * R * L * 4, dtype=torch.uint8, device=dev)   # four dt_low sets

    def once():
        ssm.ss2d_prologue_fwd(x, w["conv_w"], w["conv_b"], w["W_x"], w["W_dt"], R, N,
                              workspace=ws)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        once()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    e = x.element_size()
    # x read; u written [B,D,H,W]; delta [B,4,D,L], B and C [B,4,N,L] written
    nbytes = e * (2 * B * D * L + 4 * B * D * L + 2 * 4 * B * N * L)
    flops = 2.0 * B * L * (Kc * Kc * D + 4 * ((R + 2 * N) * D + D * R))
    return {"ms_per_call": round(ms, 4), "directions": 4, "dt_rank": R, "d_conv": Kc,
            "value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "tflops": flops / (ms * 1e-3) / 1e12}


# ---------------------------------------------------------------- CPU oracle
class OracleSampler:
    """The fp64 oracle, as it stands, over bounded samples of whole rows of
    the workload, rows spread over the host cores (one oracle call per row).
    The inputs are built once; each sample() is one timed run.  prefix = P
    (single / v1 / v2) makes a sample unit the first P positions of a row
    instead of the whole row, for runs of many short steps."""

    SEQ_KEYS = ("u", "u_b", "delta", "delta_b", "z", "B", "C", "B_b", "C_b")

    def __init__(self, spec, name, prefix=None, threads=None):
        import numpy as np

        import oracle
        from selective_state_space_111_b300.synth import make_inputs, seed_for
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from cases import row_slice, run_oracle
        self.spec, self.name = spec, name
        self.prefix = prefix if (prefix and spec.op != "ss2d" and prefix < spec.seq_len) else None
        self.row_slice, self.run_oracle = row_slice, run_oracle
        self.cores = threads or len(os.sched_getaffinity(0))
        self.t = make_inputs(spec, seed_for(name))
        oracle.build()
        rng = np.random.default_rng(0)
        self.rows = [(int(rng.integers(spec.B)), int(rng.integers(spec.D)))
                     for _ in range(100000)]

    def sample(self, seconds):
        spec, cores = self.spec, self.cores
        done = [0]
        lock = threading.Lock()
        deadline = time.perf_counter() + seconds

        def worker(k):
            i = k
            while i < len(self.rows):
                b, d = self.rows[i]
                ts = self.row_slice(spec, self.t, b, d)
                if self.prefix:
                    for key in self.SEQ_KEYS:
                        if ts.get(key) is not None:
                            ts[key] = ts[key][..., :self.prefix].contiguous()
                self.run_oracle(spec, ts)
                with lock:
                    done[0] += 1
                i += cores
                if time.perf_counter() >= deadline:
                    break

        t0 = time.perf_counter()
        th = [threading.Thread(target=worker, args=(k,)) for k in range(cores)]
        for x in th:
            x.start()
        for x in th:
            x.join()
        el = time.perf_counter() - t0
        frac = (self.prefix / spec.seq_len) if self.prefix else 1.0
        per_row_updates = spec.updates() / (spec.B * spec.D) * frac
        per_row_bytes = spec.algorithmic_bytes() / (spec.B * spec.D) * frac
        ups = done[0] * per_row_updates / el
        unit = ("row prefixes of %d positions" % self.prefix) if self.prefix else "whole rows"
        return {"value": round(done[0] * per_row_bytes / el / 1e9, 6), "unit": "GB/s",
                "elem_updates_per_s": float("%.4g" % ups), "cores": cores, "kind": "oracle",
                "seconds": round(el, 3),
                "sample": "%d %s (all directions, L=%d) of %s in %.2f s, one per oracle call, "
                          "%d threads" % (done[0], unit, spec.seq_len, self.name, el, cores)}


def cpu_baseline(spec, name, seconds, threads=None):
    return OracleSampler(spec, name, threads=threads).sample(seconds)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from selective_state_space_111_b300.synth import WORKLOADS
    spec = WORKLOADS[args.workload]
    t_all = time.perf_counter()
    nsteps = args.warmup + args.steps
    sampler = OracleSampler(spec, args.workload, prefix=512 if nsteps > 100 else None)
    # every step is a bounded sample: the whole run stays near a minute of
    # CPU time whatever --steps and --warmup are (at least one row per core)
    per_step = max(0.02, min(2.0, 60.0 / max(1, nsteps)))
    vals = []
    for i in range(args.warmup + args.steps):
        cb = sampler.sample(per_step)
        if i >= args.warmup:
            vals.append(cb)
    v = statistics.mean(c["value"] for c in vals)
    ups = statistics.mean(c["elem_updates_per_s"] for c in vals)
    # each step is a bounded sample of the workload: its measured wall time
    # is ms_per_step; the time the oracle would take for the whole workload
    # is extrapolated from the sample's throughput and reported beside it
    ms = statistics.mean(c["seconds"] for c in vals) * 1e3
    ms_full = spec.algorithmic_bytes() / (v * 1e9) * 1e3 if v > 0 else None
    line = {"metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference",
            "elem_updates_per_s": ups, "n_gpus": args.gpus, "host_only": True,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "step_is": "a bounded sample of the workload",
            "ms_whole_workload_extrapolated": round(ms_full, 1) if ms_full else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "op": spec.op, "batch": spec.B,
                       "d_inner": spec.D, "d_state": spec.N, "seq_len": spec.seq_len},
            "cpu_baseline": {"value": v, "unit": "GB/s", "kind": "oracle",
                             "cores": vals[0]["cores"],
                             "sample": "%d steps of ~%.2f s each; last: %s"
                                       % (args.steps, per_step, vals[-1]["sample"])},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t_all, 1)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward-pass timing (reported under 'backward')")
    ap.add_argument("--no-prologue", action="store_true",
                    help="skip the prologue timing (reported under 'prologue')")
    ap.add_argument("--no-out-proj", action="store_true",
                    help="skip the output-projection timing (reported under 'out_proj')")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--min-seconds", type=float, default=1.5,
                    help="repeat the K-step timed window until this much device time "
                         "has passed, sampling the clocks throughout")
    ap.add_argument("--alu-rates", action="store_true",
                    help="print the FMA / packed FMA / MUFU ex2 rates per SM per clock and exit")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.alu_rates:
        import torch
        torch.cuda.init()
        print(json.dumps({"alu_rates_per_sm_clock": alu_rates(),
                          "gpu": torch.cuda.get_device_name(0)}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
