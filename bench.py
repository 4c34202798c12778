"""Benchmark of the selective scan (S6) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ssm_scan_fwd call over the Mamba-1.4B-shaped prefill layer
(batch 4, seqlen 8192, dim 4096, dstate 16, bf16 I/O, fp32 state), inputs
resident in HBM (1.08 GB per step, larger than the 126 MB L2, so no flush is
needed).  Prints ONE JSON line (rank 0):

  value        scanned elements (batch*seqlen*dim) per second, all ranks
  roofline     HBM roofline of the scan kernel: compulsory bytes (x, delta, z,
               B, C read; out written) / the kernel's CUDA-event time, against
               the measured copy bandwidth of this GPU type
  sfu          the same kernel against its exponential-unit bound (one
               ex2 per (token, state) item; 32 per clock per SM on B300)
  e2e          the same metric through the public API from pinned HOST
               buffers, host->device and device->host copies inside the timing
  cpu_baseline the fp64 oracle on the host cores, on a bounded sample
  decode       the one-token state update (256 x 5120 x 16, 128 chained steps)
  bwd          the gradients of the same scan (ssm_scan_bwd: states
               recomputed, dx/ddelta/dz/dA/dB/dC/dD/dbias), time per call
  zoh          the same scan with the exact zero-order-hold input term
  lti          the time-invariant model's convolution mode (kernel + causal
               convolution) against the recurrence on the same constant inputs,
               on the Mamba-130M-shaped layer (the convolution is O(L^2))
  proj         the selection projections on the tensor cores (x_proj ->
               dt_low, B, C; dt_proj -> delta) for the same layer (d_model
               2048: dt_rank 128), against the HBM and bf16 tensor rooflines
  conv_scan    the Mamba block's causal conv (width 4, SiLU) in front of the
               same scan: fused (ssm_conv_scan_fwd, one pass) against the two
               separate calls (ssm_conv1d_fwd writing x_conv, then ssm_scan_fwd)

With --impl reference the fp64 CPU oracle is timed instead (the reference arm),
on a bounded sample of the same workload per step.

Under torchrun (N > 1) every rank scans its own independent batch (weak
scaling, no data-path collective); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_137_b300 import synth  # noqa: E402

WORKLOAD = synth.MAMBA_1P4B
DECODE = synth.DECODE
METRIC = "selective-scan elements (B*L*D)/s"
UNIT = "elements/s"
PEAK_FALLBACK_GBS = 6400.0
SFU_EX2_PER_CLK_PER_SM = 32        # measured: ex2.approx.f32 lane-ops per clock per SM on B300


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD.name,
                    help="scan workload name (default: the Mamba-1.4B layer)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip the zoh and lti sections")
    ap.add_argument("--no-proj", action="store_true")
    ap.add_argument("--conv-width", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target wall time of the oracle sample")
    ap.add_argument("--only", choices=["all", "scan", "decode", "conv", "bwd", "variants", "proj"],
                    default="all",
                    help="run only the prefill scan part or only the decode part (profiling)")
    return ap.parse_args()


def workload_by_name(name):
    for w in synth.SCAN_WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return PEAK_FALLBACK_GBS, "fallback"


# The sources that define each profiled kernel: its own header, the headers it
# includes, and the launch code.  A committed ncu summary records the hash of
# these files when it was captured; its traffic figure is used only while they
# are unchanged.
_KERNEL_SOURCES = {
    "scan_fwd": ("common.cuh", "tma.cuh", "scan_generic.cuh", "tile_io.cuh", "scan_warp.cuh",
                 "ssm_api.cu"),
    "conv_scan_fwd": ("common.cuh", "tma.cuh", "scan_generic.cuh", "tile_io.cuh",
                      "scan_ws.cuh", "ssm_api.cu"),
    "state_update": ("common.cuh", "tile_io.cuh", "decode.cuh", "ssm_api.cu"),
    "conv1d_fwd": ("common.cuh", "scan_generic.cuh", "tile_io.cuh", "conv.cuh", "ssm_api.cu"),
    "scan_bwd": ("common.cuh", "tma.cuh", "tile_io.cuh", "scan_warp.cuh", "scan_bwd.cuh", "scan_bwd_warp.cuh",
                 "ssm_api.cu"),
    "x_proj": ("common.cuh", "tma.cuh", "tile_io.cuh", "gemm.cuh", "ssm_api.cu"),
    "dt_proj": ("common.cuh", "tma.cuh", "tile_io.cuh", "gemm.cuh", "ssm_api.cu"),
    "lti_conv": ("common.cuh", "tma.cuh", "tile_io.cuh", "lti.cuh", "ssm_api.cu"),
}


def kernel_source_hash(kernel=None):
    """sha256 prefix of the kernel's defining sources (all of csrc/ when
    ``kernel`` is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_137_b300", "csrc")
    files = sorted(os.listdir(csrc)) if kernel is None else sorted(_KERNEL_SOURCES[kernel])
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of that kernel (the summary records their hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    kernel = next((k for k in sorted(_KERNEL_SOURCES, key=len, reverse=True)
                   if kernel_tag.startswith(k + "_")), None)
    if not m_hash or not m_bytes or kernel is None or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_bytes.group(1))


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- dist
def dist_init(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device=None):
    """Max of a per-rank scalar over all ranks (timing: the job takes as long
    as its slowest rank).  A scalar all-reduce, not a data-path collective."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank_step, steps, max_total_ms):
    """Weak scaling: every rank processes its own batch, so the job's
    throughput is all ranks' units over the slowest rank's time."""
    return world * units_per_rank_step * steps / (max_total_ms * 1e-3)


# ----------------------------------------------------------------------------- oracle sample
def oracle_sample_inputs(inp, w, nchan, nseq=1):
    """fp64 copies of channels [0, nchan) of sequences [0, nseq) (all tokens)."""
    import oracle  # noqa: F401  (test/baseline infrastructure only)
    sl = slice(0, nchan)
    f64 = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()
    return dict(x=f64(inp["x"][:nseq, :, sl]), delta=f64(inp["delta"][:nseq, :, sl]),
                A=f64(inp["A"][sl]), B=f64(inp["B"][:nseq]), C=f64(inp["C"][:nseq]),
                D=f64(inp["D"][sl]) if inp["D"] is not None else None,
                z=f64(inp["z"][:nseq, :, sl]) if inp["z"] is not None else None,
                delta_bias=f64(inp["delta_bias"][sl]) if inp["delta_bias"] is not None else None)


def calibrate_oracle(inp, w, target_s):
    """(channels, sequences) whose oracle run takes about target_s seconds on
    all host cores: channels of sequence 0 first, then whole sequences."""
    import oracle
    cores = os.cpu_count() or 1
    oracle.load()
    probe = min(w.dim, max(cores, 8))
    s = oracle_sample_inputs(inp, w, probe)
    t = time.perf_counter()
    oracle.scan_fwd(**s, nthreads=cores)
    dt = max(time.perf_counter() - t, 1e-6)
    per_chan = dt / probe
    nchan = int(min(w.dim, max(probe, target_s / per_chan)))
    if nchan >= cores:
        nchan = (nchan // cores) * cores
    nseq = 1
    if nchan >= w.dim:
        nchan = w.dim
        nseq = int(min(w.batch, max(1, target_s / (per_chan * w.dim))))
    return nchan, nseq, cores


def time_oracle(inp, w, target_s):
    """Run the oracle on a sample sized for about target_s seconds; returns
    (elements/s, seconds, channels, sequences, cores)."""
    import oracle
    nchan, nseq, cores = calibrate_oracle(inp, w, target_s)
    s = oracle_sample_inputs(inp, w, nchan, nseq)
    t = time.perf_counter()
    oracle.scan_fwd(**s, nthreads=cores)
    dt = time.perf_counter() - t
    return w.seqlen * nchan * nseq / dt, dt, nchan, nseq, cores


def time_oracle_single(inp, w, target_s):
    """The oracle on one host thread, on channels of sequence 0 sized for about
    target_s seconds; returns (elements/s, channels)."""
    import oracle
    oracle.load()
    probe = min(w.dim, 8)
    s = oracle_sample_inputs(inp, w, probe)
    t = time.perf_counter()
    oracle.scan_fwd(**s, nthreads=1)
    per_chan = max(time.perf_counter() - t, 1e-6) / probe
    nchan = int(min(w.dim, max(probe, target_s / per_chan)))
    s = oracle_sample_inputs(inp, w, nchan)
    t = time.perf_counter()
    oracle.scan_fwd(**s, nthreads=1)
    return w.seqlen * nchan / (time.perf_counter() - t), nchan


def cpu_model():
    try:
        for l in open("/proc/cpuinfo"):
            if l.startswith("model name"):
                return l.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle as it stands, on the host cores, each
    step a bounded sample (about 2 s) of the same workload."""
    if rank != 0:
        return
    import oracle
    w = workload_by_name(args.workload)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_scan_inputs(w, device=gen_dev)
    nchan, nseq, cores = calibrate_oracle(inp, w, 2.0)
    s = oracle_sample_inputs(inp, w, nchan, nseq)
    del inp
    for _ in range(args.warmup):
        oracle.scan_fwd(**s, nthreads=cores)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan_fwd(**s, nthreads=cores)
    el = time.perf_counter() - t
    value = w.seqlen * nchan * nseq * args.steps / el
    sample = (f"sequences 0..{nseq - 1} of {w.batch}, channels 0..{nchan - 1} of {w.dim}, "
              f"all {w.seqlen} tokens, per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "dim": w.dim,
            "dstate": w.dstate, "io": w.io, "state": "f32",
            "l2": f"inputs {w.io_bytes() / 1e9:.2f} GB per step > 126 MB L2; no flush"}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    from selective_state_space_137_b300 import binding, ops

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if args.only == "decode":
        peak, peak_kind = peaks()
        line = {"decode": run_decode(args, dev, peak, peak_kind), "source_hash": kernel_source_hash()}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.only == "proj":
        w = workload_by_name(args.workload)
        sinp = synth.make_scan_inputs(w, device=str(dev))
        line = {"proj": run_proj(args, w, dev, sinp), "source_hash": kernel_source_hash()}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.only == "variants":
        peak, peak_kind = peaks()
        w = workload_by_name(args.workload)
        inp = synth.make_scan_inputs(w, device=str(dev))
        line = {"zoh": run_zoh(args, w, inp, dev), "lti": run_lti(args, dev),
                "source_hash": kernel_source_hash()}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.only in ("conv", "bwd"):
        peak, peak_kind = peaks()
        w = workload_by_name(args.workload)
        inp = synth.make_scan_inputs(w, device=str(dev))
        part = run_conv if args.only == "conv" else run_bwd
        line = {("conv_scan" if args.only == "conv" else "bwd"): part(args, w, inp, dev, peak,
                                                                         peak_kind),
                "source_hash": kernel_source_hash()}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    w = workload_by_name(args.workload)
    import dataclasses
    wr = dataclasses.replace(w, seed=w.seed + 1000 * rank) if rank else w
    inp = synth.make_scan_inputs(wr, device=str(dev))
    out = torch.empty_like(inp["x"])
    last = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    plan = binding.ssm_scan_plan(desc)
    ws = torch.empty(max(plan.workspace, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = binding.ssm_scan_fwd(desc, inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                  inp["D"], inp["z"], inp["delta_bias"], out, last, None, ws,
                                  ws.numel(), stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_fwd")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        time.sleep(0.25)     # let the sampler start before the timed region
        ev[0].record(stream)
        for i in range(args.steps):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        time.sleep(0.15)
    barrier(world)
    # a bounded device wait that gave up leaves its launch incomplete: such a
    # run is not a measurement (read outside the timed region)
    require_device_ok(binding, "after the timed scan steps")
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    total_ms = max_over_ranks(total_ms, world, dev)
    ms = total_ms / args.steps
    value = whole_job_rate(world, w.tokens, args.steps, total_ms)

    peak, peak_kind = peaks()
    kernel_ms = float(np.mean(per))
    achieved = w.io_bytes() / (kernel_ms * 1e-3) / 1e9
    clocks = clk.summary()
    tag = "scan_fwd_" + w.name
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(tag),
                "peak_kind": peak_kind, "algorithmic_bytes_per_launch": w.io_bytes(),
                "kernel_ms": kernel_ms, "frac_of_8tbs": achieved / 8000.0,
                "kernel_launches_per_step": plan.launches}
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks["sm_mhz"] if clocks else None
    sfu = None
    if mhz:
        peak_items = SFU_EX2_PER_CLK_PER_SM * nsm * mhz * 1e6
        sfu = {"bound": "sfu", "achieved_items_per_s": w.items / (kernel_ms * 1e-3),
               "peak_items_per_s": peak_items,
               "frac": w.items / (kernel_ms * 1e-3) / peak_items,
               "basis": f"{SFU_EX2_PER_CLK_PER_SM} ex2/clk/SM x {nsm} SMs x median {mhz:.0f} MHz"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": config_of(w),
            "hbm_gbs": achieved, "gpu_launches": plan.launches * args.steps,
            "roofline": roofline, "sfu": sfu, "clocks": clocks}

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, w, inp, desc, plan, dev, world, binding)
    if not args.no_decode and args.only == "all":
        line["decode"] = run_decode(args, dev, peak, peak_kind)
    if not args.no_conv and args.only == "all":
        line["conv_scan"] = run_conv(args, w, inp, dev, peak, peak_kind)
    if not args.no_bwd and args.only == "all":
        line["bwd"] = run_bwd(args, w, inp, dev, peak, peak_kind)
    if not args.no_proj and args.only == "all":
        line["proj"] = run_proj(args, w, dev, inp)
    if not args.no_variants and args.only == "all":
        line["zoh"] = run_zoh(args, w, inp, dev)
        line["lti"] = run_lti(args, dev)
    if rank == 0 and world == 1 and not args.no_cpu:
        val, dt, nchan, nseq, cores = time_oracle(inp, w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"sequences 0..{nseq - 1} of {w.batch}, channels "
                                          f"0..{nchan - 1} of {w.dim}, all {w.seqlen} tokens "
                                          f"({dt:.1f} s wall)",
                                "cpu_model": cpu_model()}
        st_val, st_chan = time_oracle_single(inp, w, 2.0)
        line["cpu_baseline"]["single_thread"] = {
            "value": st_val, "unit": UNIT, "cores": 1,
            "sample": f"sequence 0, channels 0..{st_chan - 1}, all {w.seqlen} tokens"}
    elif rank == 0:
        line["cpu_baseline"] = None
    require_device_ok(binding, "after the other sections")
    line["device_status"] = "SSM_OK"
    line["source_hash"] = kernel_source_hash()
    if rank == 0:
        print(json.dumps(line), flush=True)


def require_device_ok(binding, where):
    """Refuse to report when any kernel's bounded wait timed out: its outputs
    are incomplete and its time is not the path's."""
    st = binding.ssm_get_device_status()
    if st != binding.SSM_OK:
        raise SystemExit(f"bench: device error word {binding.ssm_status_string(st)} {where}; "
                         "no result is printed")


def run_e2e(args, w, inp, desc, plan, dev, world, binding):
    """Same metric through the public API for host-resident data
    (ssm_scan_fwd_host): every step copies the activations x, delta, z, B, C
    from pinned host memory to the GPU and the output and final state back,
    pipelined over slices inside the call; A, D and the bias (the
    layer's parameters) stay on the GPU."""
    names = ["x", "delta", "z", "B", "C"]
    host = {k: inp[k].cpu().pin_memory() for k in names if inp[k] is not None}
    hout = torch.empty(inp["x"].shape, dtype=inp["x"].dtype, pin_memory=True)
    hlast = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, pin_memory=True)
    need = binding.ssm_scan_fwd_host_workspace_size(desc, 0)
    wsb = torch.empty(need + 256, dtype=torch.uint8, device=dev)
    ws = wsb[(256 - wsb.data_ptr() % 256) % 256:]
    stream = torch.cuda.current_stream(dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = hout.numel() * hout.element_size() + hlast.numel() * hlast.element_size()

    def step():
        st = binding.ssm_scan_fwd_host(desc, 0, host["x"], host["delta"], inp["A"], host["B"],
                                       host["C"], inp["D"], host.get("z"), inp["delta_bias"], hout,
                                       hlast, None, ws, ws.numel(), stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_fwd_host")

    steps = max(3, min(args.steps, 10))
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    total = max_over_ranks(a.elapsed_time(b), world, dev)
    # the bound: the same input bytes copied host -> device alone
    dbuf = [torch.empty_like(t, device=dev) for t in host.values()]
    a.record(stream)
    for _ in range(3):
        for dst, src in zip(dbuf, host.values()):
            dst.copy_(src, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize(dev)
    h2d_ms = a.elapsed_time(b) / 3
    return {"value": whole_job_rate(world, w.tokens, steps, total), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": total / steps, "api": "ssm_scan_fwd_host (16 MiB slices pipelined)",
            "pcie_gb_per_s": (h2d + d2h) / (total / steps * 1e-3) / 1e9,
            "h2d_copy_alone_ms": h2d_ms, "h2d_gb_per_s": h2d / (h2d_ms * 1e-3) / 1e9}


def run_conv(args, w, inp, dev, peak, peak_kind):
    """The causal conv (width K, SiLU, fp32 taps and bias) in front of the scan
    of workload w: fused conv+scan against conv1d then scan, CUDA events per
    call on the launching stream, inputs far larger than L2."""
    from selective_state_space_137_b300 import binding
    K = args.conv_width
    conv = synth.make_conv_inputs(w.batch, w.dim, K, seed=w.seed + 500, device=str(dev))
    out = torch.empty_like(inp["x"])
    xc = torch.empty_like(inp["x"])
    last = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    cst = torch.empty((w.batch, w.dim, K - 1), dtype=torch.float32, device=dev)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    cdesc = binding.make_conv_desc(K, True)
    plan = binding.ssm_scan_plan(desc)
    ws = torch.empty(max(plan.workspace, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fused():
        st = binding.ssm_conv_scan_fwd(desc, cdesc, inp["x"], conv["conv_w"], conv["conv_bias"],
                                       None, cst, inp["delta"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["z"], inp["delta_bias"], out, last, None,
                                       ws, ws.numel(), stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_conv_scan_fwd")

    def conv1d():
        st = binding.ssm_conv1d_fwd(desc, cdesc, inp["x"], conv["conv_w"], conv["conv_bias"],
                                    None, xc, cst, stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_conv1d_fwd")

    def scan():
        st = binding.ssm_scan_fwd(desc, xc, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"], out, last, None, ws, ws.numel(),
                                  stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_fwd")

    def timed(fns, steps):
        for _ in range(3):
            for f in fns:
                f()
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
              for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            for j, f in enumerate(fns):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        return [float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]))
                for j in range(len(fns))]

    steps = max(3, min(args.steps, 20))
    (fused_ms,) = timed([fused], steps)
    conv_ms, scan_ms = timed([conv1d, scan], steps)
    e = inp["x"].element_size()
    state_bytes = w.batch * w.dim * (K - 1) * 4
    conv_bytes = 2 * w.tokens * e + state_bytes + w.dim * (K + 1) * 4   # x in, x_conv out
    fused_bytes = w.io_bytes() + state_bytes + w.dim * (K + 1) * 4
    conv_gbs = conv_bytes / (conv_ms * 1e-3) / 1e9
    return {"width": K, "activation": "silu",
            "fused": {"ms": fused_ms, "elements_per_s": w.tokens / (fused_ms * 1e-3),
                      "gb_per_s": fused_bytes / (fused_ms * 1e-3) / 1e9,
                      "algorithmic_bytes_per_launch": fused_bytes,
                      "traffic": profiled_traffic("conv_scan_fwd_" + w.name)},
            "separate": {"conv1d_ms": conv_ms, "scan_ms": scan_ms, "ms": conv_ms + scan_ms,
                         "elements_per_s": w.tokens / ((conv_ms + scan_ms) * 1e-3)},
            "fused_speedup": (conv_ms + scan_ms) / fused_ms,
            "conv1d_roofline": {"bound": "hbm", "achieved": conv_gbs, "peak": peak, "unit": "GB/s",
                                "frac": conv_gbs / peak, "peak_kind": peak_kind,
                                "algorithmic_bytes_per_launch": conv_bytes,
                                "traffic": profiled_traffic("conv1d_fwd_" + w.name)}}


def _time_calls(fn, dev, steps):
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    return float(np.mean([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]))


def tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1800.0, "fallback"


def run_proj(args, w, dev, scan_inp=None):
    """x_proj and dt_proj of a Mamba layer with w's shape (dim = d_inner;
    dt_rank = d_model / 16 = dim / 32), bf16, on the tensor cores: time of the
    x_proj launch alone and of both, each against its HBM bytes and its
    tensor FLOPs."""
    from selective_state_space_137_b300 import binding
    R, N = max(8, w.dim // 32), w.dstate
    inp = synth.make_proj_inputs(w.batch, w.seqlen, w.dim, R, N, w.seed + 9, device=str(dev))
    M = w.batch * w.seqlen
    kw = dict(dtype=torch.bfloat16, device=dev)
    dt_low = torch.empty((M, R), **kw)
    Bm, Cm = torch.empty((M, N), **kw), torch.empty((M, N), **kw)
    delta = torch.empty((M, w.dim), **kw)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, False)   # raw step
    pd = binding.ssm_proj_desc(R, 0)
    stream = torch.cuda.current_stream(dev)

    def both():
        assert binding.ssm_selection_proj_fwd(desc, pd, inp["x"], inp["W_x"], inp["W_dt"], None, dt_low,
                                              Bm, Cm, delta, stream) == binding.SSM_OK

    def xonly():
        assert binding.ssm_selection_proj_fwd(desc, pd, inp["x"], inp["W_x"], None, None, dt_low, Bm,
                                              Cm, None, stream) == binding.SSM_OK

    steps = max(3, min(args.steps, 20))
    x_ms = _time_calls(xonly, dev, steps)
    all_ms = _time_calls(both, dev, steps)
    dt_ms = all_ms - x_ms
    hbm, hbm_kind = peaks()
    tc, tc_kind = tensor_peak()
    NO = R + 2 * N
    x_bytes = (M * w.dim + NO * w.dim + M * NO) * 2
    x_flops = 2.0 * M * NO * w.dim
    d_bytes = (M * R + w.dim * R + M * w.dim) * 2
    d_flops = 2.0 * M * w.dim * R

    def roof(ms, by, fl):
        gbs = by / (ms * 1e-3) / 1e9
        tfs = fl / (ms * 1e-3) / 1e12
        return {"ms": ms, "gb_per_s": gbs, "hbm_frac": gbs / hbm, "tflops": tfs,
                "tensor_frac": tfs / tc, "algorithmic_bytes": by, "flops": fl}
    xr, dr = roof(x_ms, x_bytes, x_flops), roof(dt_ms, d_bytes, d_flops)
    xr["traffic"] = profiled_traffic("x_proj_" + w.name)
    dr["traffic"] = profiled_traffic("dt_proj_" + w.name)
    res = {"workload": f"{w.name} x_proj ({M}x{w.dim} . {w.dim}x{NO}), dt_proj ({M}x{R} . {R}x{w.dim})",
           "dt_rank": R, "x_proj": xr, "dt_proj": dr, "both_ms": all_ms,
           "peaks": {"hbm_gbs": hbm, "hbm_kind": hbm_kind, "bf16_tflops": tc, "tensor_kind": tc_kind}}
    if scan_inp is not None:
        # projections + scan, the step finished in dt_proj's epilogue (bias,
        # softplus) against the raw projection with softplus and bias in the scan
        out = torch.empty_like(scan_inp["x"])
        last = torch.empty((w.batch, w.dim, N), dtype=torch.float32, device=dev)
        x3 = inp["x"]
        B3, C3 = Bm.view(w.batch, w.seqlen, N), Cm.view(w.batch, w.seqlen, N)
        d3 = delta.view(w.batch, w.seqlen, w.dim)
        sdesc = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, True)
        sdesc0 = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, False)
        pdesc0 = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, False)
        ws = torch.empty(max(binding.ssm_scan_workspace_size(sdesc), 16), dtype=torch.uint8,
                         device=dev)
        bias = scan_inp["delta_bias"]

        def fused():
            assert binding.ssm_selection_proj_fwd(desc, pd, x3, inp["W_x"], inp["W_dt"], bias, dt_low,
                                                  Bm, Cm, delta, stream) == binding.SSM_OK
            assert binding.ssm_scan_fwd(sdesc0, x3, d3, scan_inp["A"], B3, C3, scan_inp["D"],
                                        scan_inp["z"], None, out, last, None, ws, ws.numel(),
                                        stream) == binding.SSM_OK

        def unfused():
            assert binding.ssm_selection_proj_fwd(pdesc0, pd, x3, inp["W_x"], inp["W_dt"], None, dt_low,
                                                  Bm, Cm, delta, stream) == binding.SSM_OK
            assert binding.ssm_scan_fwd(sdesc, x3, d3, scan_inp["A"], B3, C3, scan_inp["D"],
                                        scan_inp["z"], bias, out, last, None, ws, ws.numel(),
                                        stream) == binding.SSM_OK
        def scan_sp():
            assert binding.ssm_scan_fwd(sdesc, x3, d3, scan_inp["A"], B3, C3, scan_inp["D"],
                                        scan_inp["z"], bias, out, last, None, ws, ws.numel(),
                                        stream) == binding.SSM_OK

        def scan_nosp():
            assert binding.ssm_scan_fwd(sdesc0, x3, d3, scan_inp["A"], B3, C3, scan_inp["D"],
                                        scan_inp["z"], None, out, last, None, ws, ws.numel(),
                                        stream) == binding.SSM_OK

        def proj_sp():
            assert binding.ssm_selection_proj_fwd(desc_sp, pd, x3, inp["W_x"], inp["W_dt"], bias,
                                                  dt_low, Bm, Cm, delta, stream) == binding.SSM_OK
        desc_sp = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, True)
        res["pipeline"] = {"step_in_dt_proj_ms": _time_calls(fused, dev, steps),
                           "step_in_scan_ms": _time_calls(unfused, dev, steps),
                           "proj_with_softplus_epilogue_ms": _time_calls(proj_sp, dev, steps),
                           "scan_with_softplus_ms": _time_calls(scan_sp, dev, steps),
                           "scan_without_softplus_ms": _time_calls(scan_nosp, dev, steps)}
        if R in (64, 128) and N == 16:
            # dt_proj fused into the scan's prologue (ssm_proj_scan_fwd): x_proj,
            # then the scan forms the raw step itself on the tensor cores
            dt3 = dt_low.view(w.batch, w.seqlen, R)

            def proj_scan():
                assert binding.ssm_proj_scan_fwd(sdesc, pd, x3, dt3, inp["W_dt"], scan_inp["A"], B3,
                                                 C3, scan_inp["D"], scan_inp["z"], bias, out, last,
                                                 None, ws, ws.numel(), stream) == binding.SSM_OK

            def xproj_then_proj_scan():
                xonly()
                proj_scan()
            res["pipeline"]["dt_proj_fused_in_scan_ms"] = _time_calls(xproj_then_proj_scan, dev, steps)
            res["pipeline"]["proj_scan_kernel_ms"] = _time_calls(proj_scan, dev, steps)
    return res


def run_zoh(args, w, inp, dev):
    """The forward scan of workload w with the exact zero-order-hold input
    term (ssm_scan_fwd_ex), beside the first-order one."""
    from selective_state_space_137_b300 import binding
    out = torch.empty_like(inp["x"])
    last = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    ws = torch.empty(max(binding.ssm_scan_workspace_size(desc), 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {"workload": w.name}
    for name in ("euler", "zoh"):
        opts = binding.make_opts(name)

        def call():
            st = binding.ssm_scan_fwd_ex(desc, opts, inp["x"], inp["delta"], inp["A"], inp["B"],
                                         inp["C"], inp["D"], inp["z"], inp["delta_bias"], out, last,
                                         None, ws, ws.numel(), stream)
            if st != binding.SSM_OK:
                raise binding.SSMError(st, "ssm_scan_fwd_ex")
        ms = _time_calls(call, dev, max(3, min(args.steps, 10)))
        res[name] = {"ms": ms, "elements_per_s": w.tokens / (ms * 1e-3)}
    return res


def run_lti(args, dev):
    """Convolution mode (ssm_lti_kernel + ssm_lti_conv_fwd) against the
    recurrence (ssm_scan_fwd with a constant step and B, C shared by all
    channels) on the Mamba-130M-shaped layer, fp32 kernel, bf16 I/O."""
    from selective_state_space_137_b300 import binding
    w = synth.MAMBA_130M
    g = torch.Generator(device=dev).manual_seed(5)
    N = w.dstate
    delta = 0.001 + 0.1 * torch.rand(w.dim, generator=g, device=dev)
    A = -torch.arange(1, N + 1, device=dev, dtype=torch.float32).repeat(w.dim, 1).contiguous()
    Bv = torch.randn(N, generator=g, device=dev)
    Cv = torch.randn(N, generator=g, device=dev)
    Bp, Cp = Bv.repeat(w.dim, 1).contiguous(), Cv.repeat(w.dim, 1).contiguous()
    x = torch.randn((w.batch, w.seqlen, w.dim), generator=g, device=dev).to(torch.bfloat16)
    K = torch.empty((w.dim, w.seqlen), dtype=torch.float32, device=dev)
    y = torch.empty_like(x)
    kdesc = binding.make_desc(1, w.seqlen, w.dim, N, torch.float32, False)
    cdesc = binding.make_desc(w.batch, w.seqlen, w.dim, 1, torch.bfloat16, False)
    stream = torch.cuda.current_stream(dev)

    def kern():
        assert binding.ssm_lti_kernel(kdesc, None, delta, A, Bp, Cp, K, stream) == binding.SSM_OK

    def conv():
        assert binding.ssm_lti_conv_fwd(cdesc, K, x, None, None, y, stream) == binding.SSM_OK

    dl = delta[None, None, :].expand(w.batch, w.seqlen, w.dim).contiguous().to(torch.bfloat16)
    Bs = Bv[None, None, :].expand(w.batch, w.seqlen, N).contiguous().to(torch.bfloat16)
    Cs = Cv[None, None, :].expand(w.batch, w.seqlen, N).contiguous().to(torch.bfloat16)
    sdesc = binding.make_desc(w.batch, w.seqlen, w.dim, N, torch.bfloat16, False)
    ws = torch.empty(max(binding.ssm_scan_workspace_size(sdesc), 16), dtype=torch.uint8, device=dev)
    last = torch.empty((w.batch, w.dim, N), dtype=torch.float32, device=dev)

    def rec():
        st = binding.ssm_scan_fwd(sdesc, x, dl, A, Bs, Cs, None, None, None, y, last, None, ws,
                                  ws.numel(), stream)
        assert st == binding.SSM_OK

    steps = max(3, min(args.steps, 10))
    k_ms, c_ms, r_ms = (_time_calls(f, dev, steps) for f in (kern, conv, rec))
    macs = w.batch * w.dim * w.seqlen * (w.seqlen + 1) / 2
    return {"workload": w.name, "kernel_ms": k_ms, "conv_ms": c_ms,
            "conv_gmac_per_s": macs / (c_ms * 1e-3) / 1e9, "recurrence_ms": r_ms,
            "note": "convolution mode is O(L^2) per channel; the recurrence O(L N)"}


def run_bwd(args, w, inp, dev, peak, peak_kind):
    """ssm_scan_bwd over workload w with a random dout (no final-state
    gradient): CUDA events per call on the launching stream."""
    from selective_state_space_137_b300 import binding
    g = torch.Generator(device=dev).manual_seed(w.seed + 77)
    dout = torch.randn(inp["x"].shape, generator=g, device=dev).to(inp["x"].dtype)
    f32 = dict(dtype=torch.float32, device=dev)
    dx, ddelta, dz = (torch.empty_like(inp["x"]) for _ in range(3))
    dA = torch.empty((w.dim, w.dstate), **f32)
    dB = torch.empty((w.batch, w.seqlen, w.dstate), **f32)
    dC = torch.empty_like(dB)
    dD, dbias = torch.empty(w.dim, **f32), torch.empty(w.dim, **f32)
    desc = binding.make_desc(w.batch, w.seqlen, w.dim, w.dstate, inp["x"].dtype)
    need = binding.ssm_scan_bwd_workspace_size(desc)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        st = binding.ssm_scan_bwd(desc, inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                  inp["D"], inp["z"], inp["delta_bias"], None, dout, None, dx,
                                  ddelta, dA, dB, dC, dD, dz, dbias, None, ws, ws.numel(), stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_bwd")

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    steps = max(3, min(args.steps, 10))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        call()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    ms = float(np.mean([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]))
    # the training pair: the forward keeps the state every 16 tokens, the
    # backward reads it instead of recomputing it
    ck = torch.empty(binding.ssm_scan_checkpoint_size(desc) // 4, dtype=torch.float32, device=dev)
    fout = torch.empty_like(inp["x"])
    flast = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    fws = torch.empty(max(binding.ssm_scan_workspace_size(desc), 16), dtype=torch.uint8, device=dev)
    need_ck = binding.ssm_scan_bwd_ex_workspace_size(desc, True)
    ws_ck = torch.empty(max(need_ck, 16), dtype=torch.uint8, device=dev)

    def fwd_train():
        st = binding.ssm_scan_fwd_train(desc, inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                        inp["D"], inp["z"], inp["delta_bias"], fout, flast, None, ck,
                                        fws, fws.numel(), stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_fwd_train")

    def bwd_ck():
        st = binding.ssm_scan_bwd_ex(desc, inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["z"], inp["delta_bias"], None, dout, None, ck, dx,
                                     ddelta, dA, dB, dC, dD, dz, dbias, None, ws_ck, ws_ck.numel(),
                                     stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_scan_bwd_ex")
    fwd_train_ms = _time_calls(fwd_train, dev, steps)
    bwd_ck_ms = _time_calls(bwd_ck, dev, steps)
    e = inp["x"].element_size()
    # read x, delta, z, dout, B, C; write dx, ddelta, dz (io) and dB, dC (fp32)
    algo = (4 + 3) * w.tokens * e + 2 * w.batch * w.seqlen * w.dstate * (e + 4)
    return {"workload": w.name, "ms": ms, "elements_per_s": w.tokens / (ms * 1e-3),
            "items_per_s": w.items / (ms * 1e-3), "workspace_bytes": need,
            "algorithmic_bytes_per_call": algo, "gb_per_s": algo / (ms * 1e-3) / 1e9,
            "hbm_frac": algo / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "ms_vs_forward_note": "forward of the same workload: roofline.kernel_ms",
            "training_pair": {"fwd_with_checkpoints_ms": fwd_train_ms,
                              "bwd_from_checkpoints_ms": bwd_ck_ms,
                              "workspace_bytes": need_ck,
                              "checkpoint_bytes": ck.numel() * 4}}


def run_decode(args, dev, peak, peak_kind):
    """The decode step of a 256 x 5120 x 16 fp32 state, 128 chained steps:
    warm (state stays in L2 between steps) and L2-flushed per step."""
    from selective_state_space_137_b300 import binding
    w = DECODE
    inp = synth.make_decode_inputs(w, device=str(dev))
    state = inp["state"].clone()
    out = torch.empty((w.batch, w.dim), dtype=inp["x"].dtype, device=dev)
    desc = binding.make_desc(w.batch, 1, w.dim, w.dstate, inp["x"].dtype)
    stream = torch.cuda.current_stream(dev)

    def one(s):
        st = binding.ssm_state_update(desc, state, inp["x"][s], inp["delta"][s], inp["A"],
                                      inp["B"][s], inp["C"][s], inp["D"], inp["z"][s],
                                      inp["delta_bias"], out, stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_state_update")

    for s in range(8):
        one(s)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s in range(w.steps):
        one(s)
    b.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = a.elapsed_time(b) / w.steps
    # the same 128-step chain captured once as a CUDA graph and replayed
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for s in range(w.steps):
                    st = binding.ssm_state_update(desc, state, inp["x"][s], inp["delta"][s],
                                                  inp["A"], inp["B"][s], inp["C"][s], inp["D"],
                                                  inp["z"][s], inp["delta_bias"], out,
                                                  torch.cuda.current_stream(dev))
                    if st != binding.SSM_OK:
                        raise binding.SSMError(st, "ssm_state_update")
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(4):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = a.elapsed_time(b) / (4 * w.steps)
    except Exception as exc:   # capture unsupported: report why, keep the rest
        graph_ms = f"graph capture failed: {exc}"
    # L2-flushed: write 512 MB between steps, time each step alone
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    times = []
    for s in range(32):
        flush.fill_(s & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one(s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    cold_ms = float(np.median(times))
    # the same after the write flush plus a read sweep of another buffer larger
    # than L2: L2 then holds clean lines, so the step does not also pay for
    # writing the flush buffer's dirty lines back to HBM
    sweep = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    ctimes_clean = []
    for s in range(32):
        flush.fill_(s & 0xFF)
        sweep.sum(dtype=torch.int64)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one(s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ctimes_clean.append(e0.elapsed_time(e1))
    del sweep
    clean_ms = float(np.median(ctimes_clean))
    by = w.step_bytes()
    # the same step with the width-4 causal conv in front (ssm_conv_state_update):
    # conv state (batch, dim, 3) fp32 read and shifted in place, taps (dim, 4)
    K = 4
    conv = synth.make_conv_inputs(w.batch, w.dim, K, seed=w.seed + 3, device=str(dev),
                                  with_state=True)
    cdesc = binding.make_conv_desc(K, True)

    def one_conv(s):
        st = binding.ssm_conv_state_update(desc, cdesc, conv["conv_state"], conv["conv_w"],
                                           conv["conv_bias"], state, inp["x"][s], inp["delta"][s],
                                           inp["A"], inp["B"][s], inp["C"][s], inp["D"], inp["z"][s],
                                           inp["delta_bias"], out, stream)
        if st != binding.SSM_OK:
            raise binding.SSMError(st, "ssm_conv_state_update")
    ctimes = []
    for s in range(32):
        flush.fill_(s & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one_conv(s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ctimes.append(e0.elapsed_time(e1))
    conv_ms = float(np.median(ctimes))
    conv_by = by + 2 * w.batch * w.dim * (K - 1) * 4 + w.dim * (K + 1) * 4
    return {"workload": w.name, "steps_chained": w.steps,
            "warm": {"ms_per_step": warm_ms, "gb_per_s": by / (warm_ms * 1e-3) / 1e9,
                     "steps_per_s": 1e3 / warm_ms},
            "warm_graph": ({"ms_per_step": graph_ms, "gb_per_s": by / (graph_ms * 1e-3) / 1e9,
                            "steps_per_s": 1e3 / graph_ms} if isinstance(graph_ms, float)
                           else graph_ms),
            "flushed": {"ms_per_step": cold_ms, "gb_per_s": by / (cold_ms * 1e-3) / 1e9,
                        "steps_per_s": 1e3 / cold_ms},
            "flushed_clean_l2": {"ms_per_step": clean_ms, "gb_per_s": by / (clean_ms * 1e-3) / 1e9,
                                 "frac": by / (clean_ms * 1e-3) / 1e9 / peak,
                                 "note": "write flush then a read sweep: no dirty lines to write back"},
            "conv_step_flushed": {"ms_per_step": conv_ms,
                                  "gb_per_s": conv_by / (conv_ms * 1e-3) / 1e9,
                                  "algorithmic_bytes": conv_by, "width": K},
            "roofline": {"bound": "hbm", "achieved": by / (cold_ms * 1e-3) / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": by / (cold_ms * 1e-3) / 1e9 / peak,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": by,
                         "traffic": profiled_traffic("state_update_" + w.name)}}


def main():
    args = parse()
    world, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
