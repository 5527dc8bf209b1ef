"""Benchmark of the Muon step on one rank's batch of MoE expert matrices.

Workload (per GPU): 32 experts of the model-configuration table of "Training a
1T-Parameter MoE on EU public infrastructure with PyTorch and TorchTitan"
(hidden 6144, expert hidden 1792): 64 matrices stored 6144 x 1792 (w1, w3) and
32 stored 1792 x 6144 (w2), bf16 gradients N(0,1) times a per-row log-normal
factor, fp32 momentum, bf16 parameters.  One step = momentum over all 96
matrices, the batched Newton-Schulz iteration per stored shape (5 quintic
steps) and the parameter update: the whole path.  By default each shape group
is one fused call (muon_step_batched: momentum with the norm's sum of squares,
then the iterations, the last of which writes the updated parameters);
``--path unfused`` times the three separate calls instead.  Each rank owns whole matrices
(section "FlexShard: Muon without communication"), so ranks share nothing and
the scaling is weak: N GPUs process N x 96 matrices per step.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon NS step: 1792×6144 expert matrices/s; TFLOP/s vs GB300 bf16 tensor peak"
UNIT = "matrices/s"
WORKLOAD = "rank_expert_batch_96: 64 x 6144x1792 (w1,w3) + 32 x 1792x6144 (w2) bf16, fp32 momentum, 5 quintic NS steps"
QUINTIC = (3.4445, -4.7750, 2.0315)
MU, LR, WD, EPS = 0.95, 0.02, 0.1, 1e-7
M_EXP, N_EXP = 1792, 6144
# algorithmic work per 1792 x 6144 matrix and NS iteration (symmetry-aware):
# A = X X^T takes m^2 n, B = bA + cAA takes m^3, X' = aX + BX takes 2 m^2 n
FLOPS_SYRK = M_EXP * M_EXP * N_EXP
FLOPS_POLY = M_EXP ** 3
FLOPS_AXPY = 2 * M_EXP * M_EXP * N_EXP
FLOPS_NS = 5 * (FLOPS_SYRK + FLOPS_POLY + FLOPS_AXPY)        # 3.247e11
FLOPS_NS_DENSE = 5 * (4 * M_EXP * M_EXP * N_EXP + 2 * M_EXP ** 3)
KERNEL_FLOPS = {"ns_syrk_tc": FLOPS_SYRK, "ns_poly_tc": FLOPS_POLY, "ns_axpy_tc": FLOPS_AXPY,
                "ns_axpy_apply_tc": FLOPS_AXPY}
PER_MATRIX_ELEMS = M_EXP * N_EXP
# algorithmic HBM bytes per element of the elementwise kernels
KERNEL_BYTES = {"momentum_bf16": 12, "momentum_norm_bf16": 12, "apply_bf16": 6, "norm_partial": 2, "transpose": 4}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def max_over_ranks(dist, value):
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def rank_seed_base(rank):
    """Seed base of the matrices a rank owns: every rank draws its own experts."""
    return 1234 + 3000 + 7919 * rank


def aggregate_value(matrices_per_rank, world, ms_per_step_max):
    """Whole-job matrices/s: all ranks' matrices over the slowest rank's step time."""
    return matrices_per_rank * world / (ms_per_step_max / 1e3)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ns_axpy_traffic.json")
KERNEL_SOURCE = os.path.join(ROOT, "muon_newton_schulz_expert_gb300", "csrc", "gemm_tc.cu")


def source_sha256():
    import hashlib
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def axpy_traffic_per_matrix():
    """DRAM bytes per matrix of ns_axpy_tc from the committed capture record
    (written by --ingest-ncu), or None when the kernel source changed after
    the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != source_sha256():
        return None
    return int(rec["traffic_bytes_per_matrix"])


def ingest_ncu(csv_path, matrices, command):
    """Writes profiles/ns_axpy_traffic.json from an ncu raw-page CSV
    (ncu -i <rep> --page raw --csv) of ns_gemm_kernel<2,...> (aX + BX) launches
    that each processed `matrices` matrices."""
    import csv
    with open(csv_path, newline="") as f:
        rows = list(csv.reader(f))
    head = rows[0]
    name_col = head.index("Kernel Name")
    rd, wr = head.index("dram__bytes_read.sum"), head.index("dram__bytes_write.sum")
    units = rows[1]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}

    def val(row, col):
        return float(row[col].replace(",", "")) * scale.get(units[col], 1)

    launches = [r for r in rows[2:] if len(r) > wr and "ns_gemm_kernel<2" in r[name_col]]
    if not launches:
        raise SystemExit("no ns_gemm_kernel<2,...> (aX + BX) launch in " + csv_path)
    per_launch = [val(r, rd) + val(r, wr) for r in launches]
    rec = {"kernel": "ns_axpy_tc (ns_gemm_kernel<2,...>)", "launches": len(launches), "matrices_per_launch": matrices,
           "dram_bytes_per_launch": [int(x) for x in per_launch],
           "traffic_bytes_per_matrix": int(sum(per_launch) / len(per_launch) / matrices),
           "source": os.path.relpath(KERNEL_SOURCE, ROOT), "source_sha256": source_sha256(), "command": command}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm
def run_gpu(args):
    import torch

    import muon_newton_schulz_expert_gb300 as mk
    from muon_newton_schulz_expert_gb300 import build as mkbuild
    import workloads

    rank, world, local = dist_env()
    dist = init_dist(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mkbuild.build()
    mk.lib()

    if args.workload == "profile8":   # small case for ncu captures: 8 w2-shaped matrices (176 MB, > L2)
        groups = [(8, workloads.EXPERT_HIDDEN, workloads.HIDDEN)]
    else:
        groups = [(64, workloads.HIDDEN, workloads.EXPERT_HIDDEN), (32, workloads.EXPERT_HIDDEN, workloads.HIDDEN)]
    total = sum(c for c, _, _ in groups)
    numel = total * PER_MATRIX_ELEMS
    seed0 = rank_seed_base(rank)

    def split(flat):
        views, off = [], 0
        for c, r, k in groups:
            views.append(flat[off:off + c * r * k].view(c, r, k))
            off += c * r * k
        return views

    params = torch.empty(numel, dtype=torch.bfloat16, device=dev)
    for i, (v, (c, r, k)) in enumerate(zip(split(params), groups)):
        v.copy_(workloads.parameters(c, r, k, seed0 + 10 * i + 1, device=dev))
    grads = []
    for s in range(2):   # two gradient sets alternate between steps
        g = torch.empty(numel, dtype=torch.bfloat16, device=dev)
        for i, (v, (c, r, k)) in enumerate(zip(split(g), groups)):
            v.copy_(workloads.gradients(c, r, k, seed0 + 100000 * s + 10 * i, device=dev))
        grads.append(g)
    momentum = torch.zeros(numel, dtype=torch.float32, device=dev)
    fused = args.path == "fused"
    upd = None if fused else torch.empty(numel, dtype=torch.bfloat16, device=dev)
    p_views, m_views = split(params), split(momentum)
    g_views = [split(g) for g in grads]
    u_views = None if fused else split(upd)
    # one workspace, sized for the largest group, serves every fused call (all on one stream)
    ws = torch.empty(max(mk.muon_step_workspace_bytes(c, r, k) for c, r, k in groups), dtype=torch.uint8,
                     device=dev) if fused else None
    stream = torch.cuda.current_stream(dev)

    def fused_group(p, g, m, param_free=None):
        mk.muon_step_batched(p, g, m, mu=MU, nesterov=True, steps=5, coeffs=QUINTIC, eps=EPS, lr=LR,
                             weight_decay=WD, scale=0.0, workspace=ws, stream=stream, param_free=param_free)

    def step(k):
        if fused:
            for p, g, m in zip(p_views, g_views[k % 2], m_views):
                fused_group(p, g, m)
            return
        mk.muon_momentum_update(grads[k % 2], momentum, upd, MU, True, stream)
        for u in u_views:
            mk.muon_ns_batched(u, 5, QUINTIC, EPS, stream)
        for p, u in zip(p_views, u_views):
            mk.muon_apply_update(p, u, LR, WD, 0.0, stream)

    for k in range(args.warmup):
        step(k)
    if mk.muon_get_device_status() != 0:
        raise RuntimeError("device status not OK after warm-up")
    torch.cuda.synchronize(dev)
    barrier(dist)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    launches0 = mk.muon_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mk.muon_trace_begin()
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for k in range(args.steps):
        step(k)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    trace = mk.muon_trace_end()
    launches = mk.muon_launch_count() - launches0
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    barrier(dist)
    ms_max = max_over_ranks(dist, ms)
    if mk.muon_get_device_status() != 0:
        raise RuntimeError("device status not OK after the timed steps")

    # end to end: every step's gradients come from pinned host memory and its
    # updated parameters go back to pinned host memory.  The copies run on two
    # side streams, ordered by events: the gradients of step k+1 are copied in
    # once step k's momentum kernel has consumed the device buffer, and step
    # k's parameters are copied out before step k+1's update overwrites them.
    e2e = None
    if not args.no_e2e:
        host_g = torch.empty(numel, dtype=torch.bfloat16, pin_memory=True)
        host_g.copy_(grads[0].cpu())
        host_p = torch.empty(numel, dtype=torch.bfloat16, pin_memory=True)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        g_dev = grads[0]

        host_p_views = split(host_p)

        host_g_views = split(host_g)

        def e2e_steps_fused(n):
            # step k's gradients arrive in device buffer k % 2, copied in group
            # by group while step k-1 computes (group j's call waits only for
            # its own gradients); group j's parameters are copied out while the
            # next group computes, and in step k+1's call for group j only the
            # launch that writes the parameters waits for that copy
            ev_in, ev_used, ev_out = [None, None], [None, None], [None] * len(groups)

            def copy_in(k):
                i = k % 2
                if ev_used[i] is not None:
                    s_in.wait_event(ev_used[i])
                else:
                    s_in.wait_stream(stream)
                evs = []
                for j in range(len(groups)):
                    with torch.cuda.stream(s_in):
                        g_views[i][j].copy_(host_g_views[j], non_blocking=True)
                    evs.append(s_in.record_event())
                ev_in[i] = evs

            copy_in(0)
            for k in range(n):
                i = k % 2
                if k + 1 < n:
                    copy_in(k + 1)
                for j, (p, g, m) in enumerate(zip(p_views, g_views[i], m_views)):
                    stream.wait_event(ev_in[i][j])
                    fused_group(p, g, m, param_free=ev_out[j])
                    s_out.wait_event(stream.record_event())
                    with torch.cuda.stream(s_out):
                        host_p_views[j].copy_(p, non_blocking=True)
                    ev_out[j] = s_out.record_event()
                ev_used[i] = stream.record_event()
            for e in ev_out:
                stream.wait_event(e)

        def e2e_steps_unfused(n):
            s_in.wait_stream(stream)
            with torch.cuda.stream(s_in):
                g_dev.copy_(host_g, non_blocking=True)
            ev_in = s_in.record_event()
            ev_out = None
            for k in range(n):
                stream.wait_event(ev_in)
                mk.muon_momentum_update(g_dev, momentum, upd, MU, True, stream)
                ev_mom = stream.record_event()
                if k + 1 < n:
                    s_in.wait_event(ev_mom)
                    with torch.cuda.stream(s_in):
                        g_dev.copy_(host_g, non_blocking=True)
                    ev_in = s_in.record_event()
                for u in u_views:
                    mk.muon_ns_batched(u, 5, QUINTIC, EPS, stream)
                if ev_out is not None:
                    stream.wait_event(ev_out)
                for pv, u in zip(p_views, u_views):
                    mk.muon_apply_update(pv, u, LR, WD, 0.0, stream)
                s_out.wait_event(stream.record_event())
                with torch.cuda.stream(s_out):
                    host_p.copy_(params, non_blocking=True)
                ev_out = s_out.record_event()
            stream.wait_event(ev_out)

        e2e_steps = e2e_steps_fused if fused else e2e_steps_unfused
        e2e_steps(2)
        torch.cuda.synchronize(dev)
        barrier(dist)
        ke = max(3, args.steps // 2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_steps(ke)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / ke)
        e2e = {"value": round(aggregate_value(total, world, e_ms), 3), "unit": UNIT, "ms_per_step": round(e_ms, 3),
               "h2d_bytes_per_step": numel * 2, "d2h_bytes_per_step": numel * 2, "steps": ke,
               "copies": "pinned host, side streams overlapped with compute"}

    host_res = None if args.no_host_resident else bench_host_resident(mk, torch, dev, stream, params, grads[0],
                                                                          groups, split, total, world, dist,
                                                                          max(3, args.steps // 3))
    peaks, peak_src = load_peaks()
    adamw = None if args.no_adamw else bench_adamw(mk, torch, dev, stream, float(peaks.get("hbm_gbs", 6800.0)))
    dense_ovl = None if (args.no_dense or world > 1) else bench_dense_overlap(mk, torch, dev, stream, step)
    kernels = {}
    for name, (n, t) in sorted(trace.items()):
        ent = {"launches": n, "avg_ms": round(t / n, 4), "share": None}
        if name in KERNEL_FLOPS:   # each launch covers one shape group
            flops = KERNEL_FLOPS[name] * n * total / len(groups)
            ent["tflops"] = round(flops / (t / 1e3) / 1e12, 1)
        if name in KERNEL_BYTES:
            passes = 2 if name == "transpose" else 1
            ntr = sum(c for c, r, k in groups if r > k)
            nbytes = KERNEL_BYTES[name] * PER_MATRIX_ELEMS * args.steps * (total if name != "transpose" else ntr * passes)
            ent["gbs"] = round(nbytes / (t / 1e3) / 1e9, 1)
        kernels[name] = ent
    traced_ms = sum(t for _, t in trace.values())
    for name, (n, t) in trace.items():
        kernels[name]["share"] = round(t / traced_ms, 4) if traced_ms else None
    ns_ms = sum(trace.get(k, (0, 0.0))[1] for k in ("ns_syrk_tc", "ns_poly_tc", "ns_axpy_tc", "ns_axpy_apply_tc",
                                                        "norm_partial", "norm_final", "transpose")) / args.steps
    dom = max(KERNEL_FLOPS, key=lambda k: trace.get(k, (0, 0.0))[1])
    dn, dt = trace[dom]
    achieved = KERNEL_FLOPS[dom] * dn * total / len(groups) / (dt / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    traffic = args.traffic
    if traffic is None and dom == "ns_axpy_tc" and axpy_traffic_per_matrix():
        traffic = axpy_traffic_per_matrix() * total / len(groups)   # bytes per average launch
    roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "traffic_note": "ncu dram read+write bytes per matrix (profiles/ns_axpy_traffic.json, 8-matrix "
                            "capture) x matrices per launch; null when the kernel source changed since",
            "peak_source": f"bf16_tflops_sustained ({peak_src})",
            "avg_launch_ms": round(dt / dn, 4), "launches": dn}
    tc_ms = sum(trace.get(k, (0, 0.0))[1] for k in KERNEL_FLOPS) / args.steps
    value = aggregate_value(total, world, ms_max)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the pages' expert matrices)",
        "config": {"workload": WORKLOAD if args.workload == "rank96" else
                   "profile8: 8 x 1792x6144 bf16 (ncu capture case, not a bench line)", "matrices_per_gpu": total, "ns_steps": 5, "coeffs": list(QUINTIC),
                   "mu": MU, "lr": LR, "weight_decay": WD, "eps": EPS,
                   "step_path": ("fused: muon_step_batched per shape group" if fused else
                                 "unfused: momentum, muon_ns_batched per shape group, update"),
                   "l2": "inputs larger than L2 (2.1 GB bf16 gradients + 4.2 GB fp32 momentum per step)",
                   "parallelism": f"whole-matrix ownership, {world} independent replica(s), no collective"},
        "ns_tflops": round(total * FLOPS_NS / (ns_ms / 1e3) / 1e12, 1) if ns_ms else None,
        "step_tflops": round(total * FLOPS_NS / (ms / 1e3) / 1e12, 1),
        "tensor_kernels_tflops": round(total * FLOPS_NS / (tc_ms / 1e3) / 1e12, 1) if tc_ms else None,
        "flops_per_matrix": {"algorithmic_symmetric": FLOPS_NS, "dense_equivalent": FLOPS_NS_DENSE},
        "roofline": roof, "kernels": kernels, "gpu_launches": launches, "clocks": clk, "e2e": e2e,
        "adamw": adamw, "host_resident": host_res, "dense_overlap": dense_ovl,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def bench_host_resident(mk, torch, dev, stream, params, grads, groups, split, total, world, dist, steps):
    """The step with parameters, gradients and momentum in pinned host memory
    (the pages' CPU-offload setting), streamed through the GPU by
    muon_step_host_grouped: 8 bytes per element in (bf16 gradient and parameter, fp32
    momentum) and 6 out (parameter and momentum) every step."""
    numel = params.numel()
    ph = params.cpu().pin_memory()
    gh = grads.cpu().pin_memory()
    mh = torch.zeros(numel, dtype=torch.float32).pin_memory()
    p_views, g_views, m_views = split(ph), split(gh), split(mh)

    def one():
        # both shape groups in one pipeline, so the host link does not drain between them
        mk.muon_step_host_grouped(list(zip(p_views, g_views, m_views)), mu=MU, steps=5, coeffs=QUINTIC, eps=EPS,
                                  lr=LR, weight_decay=WD, chunk=8, stream=stream)

    one()
    torch.cuda.synchronize(dev)
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1) / steps)
    del ph, gh, mh
    return {"value": round(aggregate_value(total, world, ms), 3), "unit": UNIT, "ms_per_step": round(ms, 3),
            "steps": steps, "h2d_bytes_per_step": numel * 8, "d2h_bytes_per_step": numel * 6, "chunk": 8,
            "api": "muon_step_host_grouped (pinned host parameters, gradients and momentum; both shape groups "
                   "in one pipeline)"}


def bench_dense_overlap(mk, torch, dev, stream, expert_step, reps=3):
    """The dense matrices' step beside the experts' one (section "FlexShard:
    Muon without communication": the dense matrices' Newton-Schulz runs on
    their owner ranks, overlapped with the experts').  The dense workload is
    the attention-like one (8 x 6144x6144 + 4 x 6144x1024, bf16, fp32
    momentum), sharded over one rank here, so dense_step runs no collective:
    it stacks each shape and makes one batched Newton-Schulz call per shape.
    Times, with CUDA events on the main stream: the experts' step alone, the
    dense step alone, the two one after the other on one stream, and the dense
    step on a side stream while the experts' step runs on the main one."""
    import workloads
    from muon_newton_schulz_expert_gb300 import dense

    shapes = [(workloads.HIDDEN, workloads.HIDDEN)] * 8 + [(workloads.HIDDEN, 1024)] * 4
    params = [workloads.parameters(1, r, c, 8800 + i, device=dev)[0] for i, (r, c) in enumerate(shapes)]
    grads = [workloads.gradients(1, r, c, 8900 + i, device=dev, kind="normal")[0] for i, (r, c) in enumerate(shapes)]
    moms = [torch.zeros(r, c, device=dev) for r, c in shapes]
    side = torch.cuda.Stream(dev)

    def dense_once(st):
        dense.dense_step(params, grads, moms, shapes, lr=LR, weight_decay=WD, stream=st)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    def both_overlapped():
        side.wait_stream(stream)
        expert_step(0)
        dense_once(side)
        stream.wait_stream(side)

    expert_step(0)
    dense_once(stream)
    torch.cuda.synchronize(dev)
    t_e = timed(lambda: expert_step(0))
    t_d = timed(lambda: dense_once(stream))
    t_seq = timed(lambda: (expert_step(0), dense_once(stream)))
    t_ovl = timed(both_overlapped)
    if mk.muon_get_device_status() != 0:
        raise RuntimeError("device status not OK after the dense overlap measurement")
    del params, grads, moms
    return {"dense_workload": "8 x 6144x6144 + 4 x 6144x1024 bf16 (dense_step, one rank: no collective)",
            "expert_step_ms": round(t_e, 3), "dense_step_ms": round(t_d, 3), "sequential_ms": round(t_seq, 3),
            "overlapped_ms": round(t_ovl, 3), "overlap_saving": round(1.0 - t_ovl / t_seq, 4),
            "timing": f"best of {reps}, CUDA events on the main stream"}


def bench_adamw(mk, torch, dev, stream, hbm_peak, steps=10, warmup=3):
    """AdamW on an embedding-shaped table (vocabulary 256000 x hidden 6144 of the
    model-configuration table): bf16 parameters and gradients, fp32 moments.
    22 algorithmic HBM bytes per element (read W, g, m, v; write W, m, v)."""
    numel = 256000 * 6144
    gen = torch.Generator(device=dev)
    gen.manual_seed(97)
    W = (torch.randn(numel, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    g = (torch.randn(numel, generator=gen, device=dev) * 1e-2).to(torch.bfloat16)
    m = torch.zeros(numel, device=dev)
    v = torch.zeros(numel, device=dev)
    for t in range(1, warmup + 1):
        mk.muon_adamw_update(W, g, m, v, t, stream=stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(warmup + 1, warmup + steps + 1):
        mk.muon_adamw_update(W, g, m, v, t, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    gbs = 22 * numel / (ms / 1e3) / 1e9
    del W, g, m, v
    return {"workload": "embedding table 256000x6144, bf16 params/grads, fp32 moments (inputs > L2)",
            "ms_per_update": round(ms, 4), "achieved": round(gbs, 1), "unit": "GB/s", "bound": "hbm",
            "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4), "bytes_per_element": 22}


# ----------------------------------------------------------------------------- the oracle on the host cores
def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def oracle_sample(rank_seed=0):
    """One w1-shaped (6144 x 1792) and one w2-shaped (1792 x 6144) matrix with full step inputs."""
    import torch
    import workloads
    out = []
    for i, (r, c) in enumerate(((workloads.HIDDEN, workloads.EXPERT_HIDDEN), (workloads.EXPERT_HIDDEN, workloads.HIDDEN))):
        g = workloads.gradients(1, r, c, 9000 + rank_seed + i).float().numpy()
        w = workloads.parameters(1, r, c, 9100 + rank_seed + i).float().numpy()
        out.append((g, w))
    return out


def oracle_step_matrix(g, w):
    import numpy as np
    from oracle import muon_oracle as O
    buf = np.zeros_like(g, dtype=np.float32)
    return O.muon_step(w, g, buf, mu=MU, lr=LR, weight_decay=WD, eps=EPS)


def cpu_baseline(seconds):
    sample = oracle_sample()
    t0 = time.perf_counter()
    done = 0
    while True:
        for g, w in sample:
            oracle_step_matrix(g, w)
            done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done / dt, 4), "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{done} matrices (alternating 6144x1792 and 1792x6144), full step (momentum, 5 NS steps, "
                      f"update) in fp64 numpy, {dt:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    sample = oracle_sample()
    for k in range(args.warmup):
        oracle_step_matrix(*sample[k % 2])
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle_step_matrix(*sample[k % 2])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cores = oracle_threads()
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the pages' expert matrices)",
        "config": {"workload": WORKLOAD, "reference": "fp64 CPU oracle; each step is one matrix of the workload"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} single-matrix steps alternating 6144x1792 / 1792x6144"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adamw", action="store_true", help="skip the AdamW (routers/embeddings) measurement")
    ap.add_argument("--no-host-resident", action="store_true", help="skip the host-resident state measurement")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="rank96", choices=["rank96", "profile8"],
                    help="rank96: the 96-matrix bench workload; profile8: 8 matrices for ncu captures")
    ap.add_argument("--path", default="fused", choices=["fused", "unfused"],
                    help="fused: one muon_step_batched call per shape group; unfused: the three separate calls")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture, if current")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-matrix overlap measurement")
    ap.add_argument("--ingest-ncu", metavar="CSV", default=None,
                    help="write profiles/ns_axpy_traffic.json from an ncu raw-page CSV of aX + BX launches, then exit")
    ap.add_argument("--ingest-matrices", type=int, default=8, help="matrices per captured launch (--ingest-ncu)")
    ap.add_argument("--ingest-command", default="", help="the capture's command line, recorded with the figures")
    args = ap.parse_args()
    if args.ingest_ncu:
        ingest_ncu(args.ingest_ncu, args.ingest_matrices, args.ingest_command)
        return
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
