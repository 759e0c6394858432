"""Benchmark of the selective-scan hot path: one training step = ss_fwd_save
(forward, keeping the backward's restart states) + ss_bwd_saved (backward)
over one batch of the Mamba-2.8B-layer workload (Bsz=4, L=4096, Dch=5120,
N=16, bf16 I/O, f32 state and gradients), through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is whole-job throughput in B*L*D
elements per second of forward+backward with inputs resident in HBM;
``e2e`` is the same metric with host<->device copies of each step's inputs
and results inside the timed region.  ``--impl reference`` times the CPU
oracle (the plain f64 reference the tests compare against) on a bounded
sample of the same workload on this host's cores.  Under torchrun every rank
runs an independent replica (the scan shards over batch and channels with no
exchange); rank 0 reports.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mamba_selective_scan_fwd_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "selective-scan fwd+bwd elements/s (B·L·D) and HBM GB/s vs GB300 peak"
UNIT = "elements/s"
WORKLOAD = WORKLOADS[3]  # mamba2.8b-layer-bf16: the workload the metric is quoted on


def pick_workload(name):
    """The workload named on the command line (every one runs forward + backward here)."""
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name!r}; one of {[w.name for w in WORKLOADS]}")

# Algorithmic bytes per element (B*L*D unit) for bf16 I/O, f32 gradients:
#   forward  = u, delta, z read + y write (4 x 2 B) = 8 B  (+ B, C, A, D, bias, last_state: per-(b,t) / per-d terms)
#   backward = u, delta, z, dy read (4 x 2 B) + du, ddelta, dz write (3 x 4 B) = 20 B  (+ B, C, dB, dC, dA, ...)
# The small per-(b, t, n) and per-(d, n) terms are added exactly below.


IO_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


def algorithmic_bytes(w):
    e = IO_BYTES[w.io]
    bld, bln, dn, d = w.Bsz * w.L * w.Dch, w.Bsz * w.L * w.N, w.Dch * w.N, w.Dch
    fwd = 4 * bld * e + 2 * bln * e + 4 * (dn + 2 * d) + 4 * w.Bsz * w.Dch * w.N
    bwd = 4 * bld * e + 3 * bld * 4 + 2 * bln * (e + 4) + 8 * (dn + 2 * d)
    return fwd, bwd


def mufu_counts(w):
    """MUFU operations of one call of each direction on workload w (softplus on,
    z given): the scan's ex2 per (t, d, n), which the roofline counts, and all
    of them -- per (t, d) the forward's softplus (ex2, rcp) and gate sigmoid
    (ex2, rcp), the backward's softplus with its derivative (ex2, two rcp) and
    gate sigmoid (ex2, rcp).  The chunk summaries of time-cut units, which
    walk their decays once more, are not counted."""
    return {"scan_ex2_per_direction": w.bld * w.N, "fwd_all": w.bld * (w.N + 4), "bwd_all": w.bld * (w.N + 5)}


# DRAM bytes (read + write) of the timed kernels' main passes on this workload
# (the sum over the launches of one pass: one per plan segment), from one ncu
# capture (profiles/ holds the summaries and the commands), and the digest of
# the kernel sources they were taken on: a source change since then makes the
# figure stale, and it is reported as null.
TRAFFIC = {
    # both launches of the main pass (608 one-chunk units; 32 units x 19 chunks)
    ("k_bwd2_main", "mamba2.8b-layer-bf16"): 3626368256,  # 2233.0 + 119.1 MB read, 1241.8 + 32.5 MB written
    ("k_fwd2_y", "mamba2.8b-layer-bf16"): 2228526336,     # 479.7 + 26.8 MB read, 1690.9 + 31.1 MB written
}
TRAFFIC_SRC_DIGEST = "2a8d031df0ea7598"


def measured_traffic(kernel, w):
    from mamba_selective_scan_fwd_gb300 import build

    if TRAFFIC_SRC_DIGEST is None or build.source_digest() != TRAFFIC_SRC_DIGEST:
        return None
    return TRAFFIC.get((kernel, w.name))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# MUFU ex2 results per clock per SM on GB300 (sm_103a), measured by a
# dependent-free ex2.approx.f32 throughput loop; the SFU roofline of the scan
# is B*L*D*N exponentials per direction at SMs x this rate x SM clock.
EX2_PER_CLK_PER_SM = 32.0


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 8:
                continue
            try:
                sm.append(float(row[0]))
                smax.append(float(row[1]))
            except ValueError:
                continue
            for name, val in zip(names, row[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(backend="nccl"):
    """One process per GPU (torchrun env).  Replicas only: the process group
    carries the barrier and the max-over-ranks timing, never data."""
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl" and torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms):
    """Whole-job rate: the units every replica processed over the slowest rank's time."""
    return world * units_per_rank / (ms / 1e3)


def measure_decode(dev, hbm_peak, peak_kind, steps=50):
    """One ss_decode_step per token on a Mamba-2.8B-layer decoding batch whose
    state (Bsz x Dch x N f32) is larger than the L2: HBM-bound, reported
    against the measured copy bandwidth."""
    import torch

    import mamba_selective_scan_fwd_gb300 as ss

    Bsz, Dch, N = 512, 5120, 16
    g = torch.Generator(device=dev).manual_seed(7)
    bf = torch.bfloat16
    u = torch.randn((Bsz, Dch), generator=g, device=dev).to(bf)
    delta = (0.5 * torch.randn((Bsz, Dch), generator=g, device=dev)).to(bf)
    z = torch.randn((Bsz, Dch), generator=g, device=dev).to(bf)
    Bm = torch.randn((Bsz, N), generator=g, device=dev).to(bf)
    Cm = torch.randn((Bsz, N), generator=g, device=dev).to(bf)
    A = -torch.arange(1, N + 1, device=dev, dtype=torch.float32).repeat(Dch, 1).contiguous()
    D = torch.ones(Dch, device=dev)
    bias = torch.full((Dch,), -4.0, device=dev)
    state = torch.randn((Bsz, Dch, N), generator=g, device=dev)
    y = torch.empty((Bsz, Dch), dtype=bf, device=dev)

    def step():
        ss.ss_decode_step(u, delta, A, Bm, Cm, D, z, bias, True, state, y=y)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    # state read + written, u / delta / z read and y written (bf16), B / C, A, D, bias
    nbytes = 2 * Bsz * Dch * N * 4 + 4 * Bsz * Dch * 2 + 2 * Bsz * N * 2 + Dch * N * 4 + 2 * Dch * 4
    ach = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"mamba2.8b-layer-decode-bf16 (Bsz={Bsz}, Dch={Dch}, N={N}, state {Bsz * Dch * N * 4 >> 20} MiB)",
            "ms_per_token": round(ms, 5), "tokens_per_s": round(Bsz / (ms / 1e3), 1),
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(ach / hbm_peak, 4), "peak_kind": f"{peak_kind} HBM copy",
                         "algorithmic_bytes": nbytes}}


def run_ours(args):
    import torch

    import mamba_selective_scan_fwd_gb300 as ss
    from mamba_selective_scan_fwd_gb300 import binding

    world, rank, local = dist_setup("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    w = pick_workload(args.workload)
    x = make_inputs(w, with_dy=True)
    io_dt = torch.bfloat16 if w.io == "bf16" else torch.float32
    io_keys = ("u", "delta", "B", "C", "z", "dy")
    host = {}
    for k, v in x.items():
        if v is None:
            continue
        t = torch.from_numpy(v)
        if k in io_keys:
            t = t.to(io_dt)
        host[k] = t.pin_memory()
    d = {k: v.to(dev, non_blocking=False) for k, v in host.items()}
    for k in ("D", "z", "delta_bias"):
        d.setdefault(k, None)
    dtid = binding.dtype_id(d["u"])
    plan = ss.plan_info(w.Bsz, w.L, w.Dch, w.N, dtid)
    ws_f = torch.empty(max(ss.fwd_workspace_bytes(w.Bsz, w.L, w.Dch, w.N, dtid), 256), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(ss.bwd_saved_workspace_bytes(w.Bsz, w.L, w.Dch, w.N, dtid), dtype=torch.uint8, device=dev)
    saved = torch.empty(ss.saved_bytes(w.Bsz, w.L, w.Dch, w.N, dtid), dtype=torch.uint8, device=dev)
    y = torch.empty((w.Bsz, w.L, w.Dch), dtype=io_dt, device=dev)
    last = torch.empty((w.Bsz, w.Dch, w.N), dtype=torch.float32, device=dev)
    grads = {}
    stream = torch.cuda.current_stream(dev)

    def fwd():
        ss.ss_fwd_save(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], w.softplus,
                       y=y, last_state=last, saved=saved, workspace=ws_f, stream=stream)

    def bwd():
        g = ss.ss_bwd_saved(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], w.softplus,
                            d["dy"], saved, out=grads, workspace=ws_b, stream=stream)
        grads.update(g)

    def step():
        fwd()
        bwd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-resident timing: exactly K steps between two events on the
    # launching stream, nothing else in between
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local if world > 1 else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()

    # ---- attribution: the same K steps again with per-call and per-kernel
    # events (the library records them between its own launches)
    nf, nb = plan["fwd_kernels"], plan["bwd_saved_kernels"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    kev_f = [[torch.cuda.Event(enable_timing=True) for _ in range(nf + 1)] for _ in range(K)]
    kev_b = [[torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)] for _ in range(K)]
    for e in [e for row in kev_f + kev_b for e in row]:
        e.record(stream)  # creates the event handles the library records
    torch.cuda.synchronize(dev)
    for i in range(K):
        evs[i][0].record(stream)
        binding.profile_events(kev_f[i])
        fwd()
        evs[i][1].record(stream)
        binding.profile_events(kev_b[i])
        bwd()
        evs[i][2].record(stream)
    binding.profile_events([])
    torch.cuda.synchronize(dev)
    total_ms = start.elapsed_time(end)
    t_fwd = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_bwd = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    # per-kernel averages: kernel j of a call runs between its events j and j + 1
    k_fwd = [sum(r[j].elapsed_time(r[j + 1]) for r in kev_f) / K for j in range(nf)]
    k_bwd = [sum(r[j].elapsed_time(r[j + 1]) for r in kev_b) / K for j in range(nb)]
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / K
    value = job_throughput(w.bld * K, world, total_ms)

    # ---- end to end through the public API with host buffers.  Every step copies
    # its inputs from pinned host memory and its outputs back; two sets of device
    # input / output buffers and one copy stream per direction let step i's
    # input copy run during step i - 1's compute and its output copy during
    # step i + 1's (the restart states and workspaces stay on the compute
    # stream).  The output copy bounds it (1178 MB per step); splitting each
    # copy over two streams per direction was no faster.
    in_keys = [k for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "dy") if k in host]
    h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
    out_host = {"y": torch.empty(y.shape, dtype=y.dtype).pin_memory(),
                "last_state": torch.empty(last.shape, dtype=last.dtype).pin_memory()}
    for k, v in grads.items():
        if v is not None:
            out_host[k] = torch.empty(v.shape, dtype=v.dtype).pin_memory()
    d2h = sum(v.numel() * v.element_size() for v in out_host.values())
    e2e_steps = max(2, min(args.e2e_steps, K))
    sets = []
    for _ in range(2):
        di = {k: (None if v is None else torch.empty_like(v)) for k, v in d.items()}
        sets.append({"d": di, "y": torch.empty_like(y), "last": torch.empty_like(last), "g": {}})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

    def e2e_run(nsteps, start_ev=None):
        if start_ev is not None:
            s_in.wait_event(start_ev)
        for i in range(nsteps):
            j = i % 2
            bs = sets[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["done"][j])  # step i - 2 is done reading this set's inputs
                for k in in_keys:
                    bs["d"][k].copy_(host[k], non_blocking=True)
                ev["in"][j].record(s_in)
            stream.wait_event(ev["in"][j])
            if i >= 2:
                stream.wait_event(ev["out"][j])  # step i - 2's outputs have left this set
            di = bs["d"]
            ss.ss_fwd_save(di["u"], di["delta"], di["A"], di["B"], di["C"], di["D"], di["z"], di["delta_bias"],
                           w.softplus, y=bs["y"], last_state=bs["last"], saved=saved, workspace=ws_f, stream=stream)
            bs["g"].update(ss.ss_bwd_saved(di["u"], di["delta"], di["A"], di["B"], di["C"], di["D"], di["z"],
                                           di["delta_bias"], w.softplus, di["dy"], saved, out=bs["g"],
                                           workspace=ws_b, stream=stream))
            ev["done"][j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["done"][j])
                out_host["y"].copy_(bs["y"], non_blocking=True)
                out_host["last_state"].copy_(bs["last"], non_blocking=True)
                for k, v in bs["g"].items():
                    if v is not None:
                        out_host[k].copy_(v, non_blocking=True)
                ev["out"][j].record(s_out)
        stream.wait_event(ev["out"][(nsteps - 1) % 2])

    e2e_run(2)
    torch.cuda.synchronize(dev)
    # three timed runs of e2e_steps steps: the host link is shared with other
    # work on the machine and its throughput varies from run to run (seen: 2x),
    # so the median is reported and every run is listed
    e2e_runs = []
    for _ in range(3):
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(e2e_steps, start_ev=e0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_runs.append(max_over_ranks(e0.elapsed_time(e1), world))
    e2e_ms = sorted(e2e_runs)[1]
    e2e_value = job_throughput(w.bld * e2e_steps, world, e2e_ms)

    # ---- roofline of the dominant kernel (the backward's main kernel) and of the forward kernel
    hbm_peak, peak_kind = load_peaks()
    fwd_bytes, bwd_bytes = algorithmic_bytes(w)
    # the main backward kernel writes everything but dB / dC and dA / dD / ddelta_bias (the reductions do)
    bwd_main_bytes = bwd_bytes - 2 * w.Bsz * w.L * w.N * 4 - 4 * (w.Dch * w.N + 2 * w.Dch)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sm_mhz = clk.get("sm_mhz") or 2070.0
    exp_peak = sms * EX2_PER_CLK_PER_SM * sm_mhz * 1e6  # ex2 / s
    exps = w.bld * w.N

    def roof(bytes_, t_ms):
        t_hbm = bytes_ / (hbm_peak * 1e9)
        t_sfu = exps / exp_peak
        if t_hbm >= t_sfu:
            ach = bytes_ / (t_ms / 1e3) / 1e9
            return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(ach / hbm_peak, 4), "peak_kind": f"{peak_kind} HBM copy",
                    "roofline_ms": round(t_hbm * 1e3, 4), "algorithmic_bytes": bytes_}
        ach = exps / (t_ms / 1e3) / 1e9
        pk = exp_peak / 1e9
        return {"bound": "alu", "achieved": round(ach, 1), "peak": round(pk, 1), "unit": "Gexp2/s",
                "frac": round(ach / pk, 4),
                "peak_kind": f"MUFU ex2: {sms} SMs x {EX2_PER_CLK_PER_SM:g}/clk x {sm_mhz:g} MHz (median sampled)",
                "roofline_ms": round(t_sfu * 1e3, 4), "algorithmic_bytes": bytes_}

    # launch order of a call: the summary passes of the chunked segments, then
    # each segment's main pass (then, in the backward, the two reductions)
    segs = plan["segments"]
    seg_tag = [f"{u} units x {k} chunk{'s' if k > 1 else ''}" for u, k in segs]
    fwd_names = ([f"k_fwd2 chunk summary ({seg_tag[i]})" for i, (_, k) in enumerate(segs) if k > 1] +
                 [f"k_fwd2 y + saved states ({t})" for t in seg_tag])
    bwd_names = ([f"k_bwd2 reverse summary ({seg_tag[i]})" for i, (_, k) in enumerate(segs) if k > 1] +
                 [f"k_bwd2 main ({t})" for t in seg_tag] + ["k_bwd2_reduce_bc", "k_bwd2_reduce_params"])
    n_sum = sum(1 for _, k in segs if k > 1)
    main_f = range(n_sum, n_sum + len(segs))  # the forward's main pass: one launch per segment
    main_b = range(n_sum, n_sum + len(segs))
    t_main_f = sum(k_fwd[j] for j in main_f)
    t_main_b = sum(k_bwd[j] for j in main_b)
    r_bwd = roof(bwd_main_bytes, t_main_b)
    r_bwd.update({"kernel": f"k_bwd2 main pass (ss_bwd_saved; {len(segs)} launch{'es' if len(segs) > 1 else ''})",
                  "ms": round(t_main_b, 4), "traffic": measured_traffic("k_bwd2_main", w)})
    r_fwd = roof(fwd_bytes, t_main_f)
    r_fwd.update({"kernel": f"k_fwd2 main pass (ss_fwd_save; {len(segs)} launch{'es' if len(segs) > 1 else ''})",
                  "ms": round(t_main_f, 4), "traffic": measured_traffic("k_fwd2_y", w)})
    t_roof = roof(fwd_bytes, t_fwd)["roofline_ms"] + roof(bwd_bytes, t_bwd)["roofline_ms"]
    kernel_ms = {n: round(v, 4) for n, v in zip(fwd_names + bwd_names, k_fwd + k_bwd)}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "Bsz": w.Bsz, "L": w.L, "Dch": w.Dch, "N": w.N, "io": w.io,
                   "terms": "D, z, delta_bias, softplus, last_state", "chunks": plan["chunks"],
                   "l2": "no flush: each step reads and writes > 2 GB, far above the 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_gbs": round((fwd_bytes + bwd_bytes) / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": r_bwd, "roofline_fwd": r_fwd,
        "roofline_step_frac": round(t_roof / ms_per_step, 4), "mufu_ops": mufu_counts(w),
        "fwd_ms": round(t_fwd, 4), "bwd_ms": round(t_bwd, 4), "kernel_ms": kernel_ms,
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "runs": [round(job_throughput(w.bld * e2e_steps, world, v), 1) for v in e2e_runs],
                "of_runs": "median"},
        "gpu_launches": K * (plan["fwd_kernels"] + plan["bwd_saved_kernels"]),  # the timed region only
    }
    if not args.no_decode:
        line["decode"] = measure_decode(dev, hbm_peak, peak_kind)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def _oracle_sample(orc, w, x, rows):
    """The oracle's forward and backward on a row sample of the workload; returns seconds."""
    t0 = time.perf_counter()
    orc.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], w.softplus, rows=rows)
    orc.bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], w.softplus, dy=x["dy"],
            rows=rows, want_dBdC=True)
    return time.perf_counter() - t0


def cpu_baseline(w, x, budget_s=15.0):
    """The oracle, as it stands, on a bounded row sample of the workload (all host cores).

    Row batches of growing size run until about ``budget_s`` seconds of oracle
    work have been timed; the rate is rows x L over the summed time."""
    import numpy as np

    import oracle

    orc = oracle.get()
    cores = oracle.default_threads()
    # f64 copies once, outside the timed sample
    x64 = {k: (None if v is None else np.ascontiguousarray(v, dtype=np.float64)) for k, v in x.items()}
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.Bsz * w.Dch)
    _oracle_sample(orc, w, x64, perm[:cores])  # untimed: first-call overheads
    done, spent, n = 0, 0.0, cores
    while spent < budget_s and done < perm.size:
        rows = perm[done:done + n]
        spent += _oracle_sample(orc, w, x64, rows)
        done += rows.size
        n = min(2 * n, perm.size - done)
    return {"value": round(done * w.L / spent, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} of {w.Bsz * w.Dch} (b, d) rows, full L={w.L}, forward + backward incl. dB/dC "
                      f"contributions, f64, {spent:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle

    w = pick_workload(args.workload)
    x = make_inputs(w, with_dy=True)
    x64 = {k: (None if v is None else np.ascontiguousarray(v, dtype=np.float64)) for k, v in x.items()}
    orc = oracle.get()
    cores = oracle.default_threads()
    rng = np.random.default_rng(1)
    # size each step's row sample so that warmup + steps fit in about two minutes
    probe = _oracle_sample(orc, w, x64, rng.choice(w.Bsz * w.Dch, cores, replace=False)) / cores
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(cores, min(w.Bsz * w.Dch, per_step_budget / max(probe, 1e-6))))
    n = max(1, n // cores * cores) if n >= cores else n
    for _ in range(args.warmup):
        _oracle_sample(orc, w, x64, rng.choice(w.Bsz * w.Dch, n, replace=False))
    total = 0.0
    for _ in range(args.steps):
        total += _oracle_sample(orc, w, x64, rng.choice(w.Bsz * w.Dch, n, replace=False))
    value = args.steps * n * w.L / total
    sample = f"{n} of {w.Bsz * w.Dch} (b, d) rows per step, full L={w.L}, forward + backward, f64 oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "Bsz": w.Bsz, "L": w.L, "Dch": w.Dch, "N": w.N, "io": w.io},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the single-step decoding measurement")
    ap.add_argument("--workload", default=WORKLOAD.name,
                    help="workload to time (default: the one the metric is quoted on)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
