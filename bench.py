#!/usr/bin/env python
"""Benchmark of the selective scan (Mamba S6) on B300: one JSON line.

A step is one selective-scan call over the whole workload (default: the long-sequence
scan, batch 1 x 1536 channels x 131072 steps x 64 states, bf16 I/O, fp32 state, final
state returned), inputs resident in HBM. `value` is scan elements (batch*dim*L*N) per
second over all ranks; each rank scans its own copy (weak scaling, no collective on the
data path). The line also carries the recurrent-step (decode) throughput, the roofline of
the step against the MUFU exp2 peak, the fp64 CPU oracle timed on this host's cores, an
end-to-end number through the host-buffer C-ABI entry point, and the SM clocks sampled
during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long128k|m130|block512]
    python bench.py --impl reference ...   # the fp64 CPU oracle on a bounded sample
    python bench.py --measure-ex2          # only the ex2 throughput probe (the roofline's peak)

The line also carries one forward-scan line per other workload (`configs`), the maximum
relative error of sampled output channels against the fp64 oracle (computed after the timed
region), and the FP32-pipe bound beside the exponential (MUFU) bound.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from selective_state_space_153_b300 import gen  # noqa: E402

SM_COUNT = 148
# MUFU ex2 lanes per SM and clock (4 sub-partitions x 8 lanes). `--measure-ex2` runs the probe
# (selective_state_space_153_b300/probe/ex2_rate.cu): independent ex2 chains, timed per SM
# with the SM's own cycle counter, measured 31.85 per SM clock on B300.
EX2_PER_CLK_SM = 32
FP32_LANES_PER_CLK_SM = 128  # FFMA lanes per SM and clock (packed f32x2 issue at the same lane rate)
FALLBACK_HBM_GBS = 6400.0

# dram__bytes_read.sum + dram__bytes_write.sum of one long-sequence scan call (aggregate pass +
# combine + full pass), from a one-pass ncu capture of the full-size call, together with the
# hash of the channel-pair kernel's sources it was taken on: a different hash (the kernels
# changed since) reports the traffic as unknown (null) rather than a stale count.
TRAFFIC_BYTES_PER_LAUNCH = {"long128k": ("37d6e199aa8ca45c", 2094964480)}   # (source hash, bytes)
TRAFFIC_SOURCES = ("scan_pair.cuh", "scan_seq.cuh", "check.cuh", "k_pair_impl.cuh", "k_seq.cu", "common.cuh",
                   "launch.h", "ptx.cuh")


def pair_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "selective_state_space_153_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    src_hash, nbytes = TRAFFIC_BYTES_PER_LAUNCH.get(workload, (None, None))
    return nbytes if (src_hash is not None and src_hash == pair_source_hash()) else None


def probe_ex2():
    """ex2 per SM and clock measured on this device by the probe library (None if unavailable)."""
    try:
        from selective_state_space_153_b300 import build
        lib = ctypes.CDLL(build.PROBE_LIB)
        lib.ssm_probe_ex2_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]
        lib.ssm_probe_ex2_rate.restype = ctypes.c_int
        r, ms = ctypes.c_double(0), ctypes.c_double(0)
        if lib.ssm_probe_ex2_rate(4096, ctypes.byref(r), ctypes.byref(ms)) != 0:
            return None
        return {"per_clk_sm": r.value, "probe_ms": ms.value,
                "how": "16 CTAs x 128 threads per SM, 32 independent ex2 chains per thread; per SM, "
                       "its CTAs' ex2 count over its first-start-to-last-end clock64 span; median over SMs"}
    except OSError:
        return None


def count_kernel_launches(fn):
    """Kernels launched by one call of fn, counted by the CUDA activity profiler (memsets and
    copies excluded). None if the profiler is unavailable."""
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        kern = [n for n in names if not n.lower().startswith(("memset", "memcpy"))]
        return len(kern), sorted(set(kern))
    except Exception:  # noqa: BLE001
        return None, []


def workload_config(args):
    from dataclasses import replace
    cfg = gen.SCAN_CONFIGS[args.workload]
    return replace(cfg, L=args.seqlen) if args.seqlen > 0 else cfg


def scan_io_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one scan call: every input read once, every output written once."""
    esz = 2 if cfg.io == "bf16" else 4
    return (cfg.Bt * cfg.D * cfg.L * esz * (3 + (1 if cfg.gate else 0))      # u, delta, (z), y
            + 2 * cfg.Bt * cfg.N * cfg.L * esz + cfg.D * cfg.N * 4 + 2 * cfg.D * 4
            + (cfg.Bt * cfg.D * cfg.N * 4 if cfg.last_state else 0))


def config_json(cfg) -> dict:
    """The bench line's `config`, identical for both arms."""
    return {"workload": f"{cfg.name}: selective scan Bt={cfg.Bt} D={cfg.D} L={cfg.L} N={cfg.N} "
                        f"io={cfg.io} gate={cfg.gate} last_state={cfg.last_state}",
            "batch": cfg.Bt, "dim": cfg.D, "seqlen": cfg.L, "dstate": cfg.N, "io": cfg.io,
            "l2": "inputs larger than L2 (%.0f MB per step)" % (scan_io_bytes(cfg) / 1e6)}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long128k", choices=list(gen.SCAN_CONFIGS))
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override the workload's sequence length (profiling of a smaller case)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-zoh", action="store_true")
    ap.add_argument("--no-struct", action="store_true", help="skip the structured-A fast-path line")
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' forward-scan lines")
    ap.add_argument("--no-check", action="store_true", help="skip the sampled oracle check of the output")
    ap.add_argument("--measure-ex2", action="store_true", help="run only the ex2 throughput probe")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": 2032.0}, "fallback"


# ---------------------------------------------------------------------------- distributed
def dist_setup(n):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def weak_scaling_value(units_per_rank, ws, max_seconds_per_step):
    """Whole-job throughput: every rank processes its own copy of the workload (weak
    scaling), so the job's units per step are ws * units_per_rank, over the slowest rank."""
    return ws * units_per_rank / max_seconds_per_step


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- clocks (NVML)
class ClockSampler:
    """Samples SM clock and clock-event reasons with nvidia-smi during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"ssm_clocks_{os.getpid()}_{cuda_index}.csv")
        try:
            props = torch.cuda.get_device_properties(cuda_index)
            self.uuid = "GPU-" + str(props.uuid)
        except Exception:  # noqa: BLE001
            self.uuid = None

    def __enter__(self):
        import subprocess
        if self.uuid is None:
            return self
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable: nvidia-smi"], "samples": 0}
        mhz, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                mhz.append(float(f[0])); mx = float(f[1]); pw.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(statistics.median(mhz)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------- oracle timing
def oracle_rate(inp, target_s, nthreads):
    """fp64 oracle on a bounded sample of channels (full sequence): elements/s."""
    import oracle
    cfg = inp["cfg"]
    f = gen.as_f64

    def run(chs):
        bs = np.array([c[0] for c in chs]); ds = np.array([c[1] for c in chs])
        rows = lambda t: None if t is None else t[torch.as_tensor(bs), torch.as_tensor(ds), :].to(torch.float64).numpy()  # noqa: E731
        args = (rows(inp["u"]), rows(inp["delta"]), f(inp["A"])[ds], f(inp["B"]), f(inp["C"]), bs)
        kw = dict(D=None if inp["D"] is None else f(inp["D"])[ds], z=rows(inp["z"]),
                  delta_bias=None if inp["delta_bias"] is None else f(inp["delta_bias"])[ds],
                  delta_softplus=inp["delta_softplus"], nthreads=nthreads)
        t = time.perf_counter()
        oracle.scan_rows(*args, **kw)
        return time.perf_counter() - t

    allch = [(b, d) for b in range(cfg.Bt) for d in range(cfg.D)]
    t1 = run(allch[:1])
    k = int(max(1, min(len(allch), round(target_s * nthreads / max(t1, 1e-6)))))
    k = max(min(k, len(allch)), 1)
    step = max(1, len(allch) // k)
    chs = allch[::step][:k]
    t = run(chs)
    elems = len(chs) * cfg.L * cfg.N
    return elems / t, len(chs), min(nthreads, len(chs)), t


# ---------------------------------------------------------------------------- our arm
def bench_ours(args, rank, ws, local):
    from selective_state_space_153_b300 import ssm
    ssm.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = workload_config(args)
    inp = gen.scan_inputs(cfg)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(g["u"])
    last = torch.empty((cfg.Bt, cfg.D, cfg.N), dtype=torch.float32, device=dev) if cfg.last_state else None
    stream = torch.cuda.current_stream()
    # The headline, the ZOH, conv-front and end-to-end lines run the general path (one
    # exponential per element, the SFU roofline's premise; the library's default). The
    # structured-A path, which the generator's A = -(n+1) would pass, is timed separately.
    ssm.set_structured_a(False)
    # The chunk-carry workspace is allocated once, outside the timed region, and passed in
    # (ssm_selective_scan_fwd_ws), so that the device times hold the scan kernels and not the
    # stream-ordered allocator; the end-to-end line keeps the allocating host entry point.
    io_code = ssm.SSM_BF16 if cfg.io == "bf16" else ssm.SSM_F32
    scan_ws = torch.empty(max(1, ssm.workspace_bytes(cfg.Bt, cfg.D, cfg.L, cfg.N, io_code)), dtype=torch.uint8,
                          device=dev)

    def step():
        ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                               delta_bias=g["delta_bias"], delta_softplus=cfg.softplus, y=y, last_state=last,
                               stream=stream, workspace=scan_ws)

    def timed(fn):
        """ms per call of fn: warm-up, then args.steps calls between events on `stream`."""
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        t0.record(stream)
        for _ in range(args.steps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        ms_ = max_over_ranks(t0.elapsed_time(t1), ws) / args.steps
        assert ssm.stream_status(stream) == ssm.SSM_OK
        return ms_

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert ssm.stream_status(stream) == ssm.SSM_OK
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    barrier(ws)
    torch.cuda.synchronize()
    with sampler:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, ws)
    assert ssm.stream_status(stream) == ssm.SSM_OK

    elems = cfg.elements
    io_bytes = scan_io_bytes(cfg)
    t_step = ms_max / args.steps / 1e3
    peaks, peak_kind = measured_peaks()
    clocks = sampler.summary()
    sm_max = float(peaks.get("sm_max_mhz", 2032.0))
    ex2_peak = SM_COUNT * EX2_PER_CLK_SM * sm_max * 1e6 / 1e9          # Gexp/s at the max SM clock
    achieved = elems / t_step / 1e9
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    launches_per_step, kernel_names = count_kernel_launches(step)
    if not launches_per_step:   # profiler unavailable (or held by another tool): the planner's count
        launches_per_step = 3 if ssm.workspace_bytes(cfg.Bt, cfg.D, cfg.L, cfg.N,
                                                    ssm.SSM_BF16 if cfg.io == "bf16" else ssm.SSM_F32) > 0 else 1
    out = {
        "metric": "scan elements/s (B*D*L*N/s); fraction of the max(HBM, SFU) roofline; decode tok/s",
        "value": weak_scaling_value(elems, ws, t_step), "unit": "elem/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded generator, PCG64)",
        "config": config_json(cfg),
        "tokens_per_s": ws * cfg.Bt * cfg.L / t_step,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": ex2_peak, "unit": "Gexp/s",
                     "frac": achieved / ex2_peak,
                     "traffic": measured_traffic(args.workload) if not args.seqlen else None,
                     "peak_source": f"MUFU ex2 {EX2_PER_CLK_SM}/clk/SM x {SM_COUNT} SMs x {sm_max:.0f} MHz",
                     "kernel": "whole scan call (%d launch%s: %s)" % (
                         launches_per_step, "es" if launches_per_step > 1 else "",
                         ", ".join(k.split("(")[0].replace("void ", "") for k in kernel_names) or "n/a"),
                     "hbm": {"achieved_gbs": io_bytes / t_step / 1e9, "peak_gbs": hbm, "peak_kind": peak_kind,
                             "frac": io_bytes / t_step / 1e9 / hbm},
                     "frac_at_sampled_clock": (achieved / (SM_COUNT * EX2_PER_CLK_SM * clocks["sm_mhz"] * 1e6 / 1e9)
                                               if clocks["sm_mhz"] else None),
                     # the second compute bound: dt*A, dt*u*B, the recurrence FMA and the readout
                     # FMA per element on the FP32 pipe (128 lanes per SM and clock)
                     "fp32_pipe": {"ops_per_element": 4,
                                   "peak_gops": SM_COUNT * FP32_LANES_PER_CLK_SM * sm_max * 1e6 / 1e9,
                                   "frac": 4 * elems / t_step / 1e9 / (SM_COUNT * FP32_LANES_PER_CLK_SM * sm_max * 1e6 / 1e9)},
                     "ex2_probe": probe_ex2()},
        "clocks": clocks,
        "gpu_launches": args.steps * launches_per_step,
        "kernels_per_step": kernel_names,
    }
    # maximum relative error of sampled channels (whole sequence) against the fp64 oracle, on
    # the output of the last timed call (outside the timed region)
    if not args.no_check and rank == 0:
        out["check"] = oracle_check(inp, y, last, cfg)
    # forward-scan lines for the other workloads (each its own inputs, timed the same way)
    if not args.no_configs:
        out["configs"] = {}
        for name, c in gen.SCAN_CONFIGS.items():
            if name == cfg.name:
                continue
            line = bench_config(c, dev, stream, timed, ex2_peak, hbm)
            out["configs"][name] = line
            out["gpu_launches"] += args.steps * line["launches_per_step"]
    # the exact zero-order-hold variant on the same workload, timed the same way
    if not args.no_zoh:
        def zstep():
            ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                   delta_bias=g["delta_bias"], delta_softplus=cfg.softplus, y=y, last_state=last,
                                   stream=stream, workspace=scan_ws, discretization="zoh")
        zms = timed(zstep)
        out["zoh"] = {"discretization": "exact zero-order hold (exp(dt*A) - 1)/A * B",
                      "ms_per_step": zms, "value": weak_scaling_value(elems, ws, zms / 1e3), "unit": "elem/s",
                      "roofline_frac": elems / (zms / 1e3) / 1e9 / ex2_peak}
        out["gpu_launches"] += args.steps * launches_per_step
    # the conv1d (K = 4) + SiLU front fused in the scan, on the same workload, timed the same way
    if not args.no_conv:
        gw = torch.Generator().manual_seed(11)
        cw = (torch.randn(cfg.D, 4, generator=gw) * 0.5).to(dev)
        cbias = (torch.randn(cfg.D, generator=gw) * 0.2).to(dev)

        cws = torch.empty(max(1, int(ssm.load().ssm_conv_selective_scan_workspace_bytes(
            ctypes.byref(ssm.dims(cfg.Bt, cfg.D, cfg.L, cfg.N, io_code))))), dtype=torch.uint8, device=dev)

        def cstep():
            ssm.conv_selective_scan_fwd(g["u"], cw, cbias, g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                        delta_bias=g["delta_bias"], delta_softplus=cfg.softplus, y=y,
                                        last_state=last, stream=stream, workspace=cws)
        cms = timed(cstep)
        out["conv_front"] = {"fused": "causal depthwise conv1d (K=4) + bias + SiLU in front of the scan",
                             "ms_per_step": cms, "value": weak_scaling_value(elems, ws, cms / 1e3), "unit": "elem/s",
                             "roofline_frac": elems / (cms / 1e3) / 1e9 / ex2_peak}
        out["gpu_launches"] += args.steps * launches_per_step
    # the structured-A fast path (run-time detected A[d, n] == (n+1)*A[d, 0]; decays from
    # powers of exp(dt*A[d, 0])) on the same workload, timed the same way; not the headline:
    # it evaluates fewer than one exponential per element
    if not args.no_struct:
        ssm.set_structured_a(True)
        sms = timed(step)
        ssm.set_structured_a(False)
        out["structured_a"] = {
            "path": "A[d,n] = (n+1)*A[d,0] detected per warp; A_bar[n] = r^(n+1), r = exp(dt*A[d,0])",
            "ms_per_step": sms, "value": weak_scaling_value(elems, ws, sms / 1e3), "unit": "elem/s",
            "speedup_vs_general": (ms_max / args.steps) / sms,
            "exps_per_element": "(1 + KS/4)/KS for KS states per lane: 3/8 at KS = 8, 1/2 at KS = 4",
            "elem_rate_over_general_sfu_bound": elems / (sms / 1e3) / 1e9 / ex2_peak}
        out["gpu_launches"] += args.steps * launches_per_step
    # end to end: host buffers through the C ABI, copies inside the timed region
    if not args.no_e2e:
        pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        yh = torch.empty_like(pin["u"]).pin_memory()
        lh = torch.empty((cfg.Bt, cfg.D, cfg.N), dtype=torch.float32).pin_memory() if cfg.last_state else None

        def host_step():
            ssm.selective_scan_fwd_host(pin["u"], pin["delta"], pin["A"], pin["B"], pin["C"], D=pin["D"], z=pin["z"],
                                        delta_bias=pin["delta_bias"], delta_softplus=cfg.softplus, y=yh,
                                        last_state=lh)
        host_step()
        ke = max(2, min(args.steps, 5))
        barrier(ws)
        t = time.perf_counter()
        for _ in range(ke):
            host_step()
        te = max_over_ranks(time.perf_counter() - t, ws)
        h2d = sum(v.numel() * v.element_size() for k, v in pin.items()
                  if isinstance(v, torch.Tensor) and k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias"))
        d2h = yh.numel() * yh.element_size() + (lh.numel() * 4 if lh is not None else 0)
        out["e2e"] = {"value": ws * elems * ke / te, "unit": "elem/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": te / ke * 1e3,
                      "entry": "ssm_selective_scan_fwd_host (pinned host buffers)"}
        del pin, yh
    if not args.no_bwd:
        out["backward"] = bench_backward(dev, ws, gen.M130)
        out["gpu_launches"] += out["backward"]["launches"]
        out["backward_long"] = bench_backward(dev, ws, gen.BWD_LONG)
        out["gpu_launches"] += out["backward_long"]["launches"]
    if not args.no_decode:
        out["decode"] = bench_decode(dev)
        out["gpu_launches"] += out["decode"]["launches"]
    if rank == 0 and ws == 1 and not args.no_cpu:
        nthreads = os.cpu_count() or 1
        rate, nch, cores, secs = oracle_rate(inp, args.cpu_seconds, nthreads)
        out["cpu_baseline"] = {"value": rate, "unit": "elem/s", "cores": cores, "kind": "oracle",
                               "sample": f"{nch} of {cfg.Bt * cfg.D} channels, full L={cfg.L}, N={cfg.N}, "
                                         f"fp64 sequential C, {cores} threads, {secs:.1f} s"}
    return out


def oracle_check(inp, y, last, cfg):
    """Max relative error (against max(|oracle|, magnitude companion)) of a few sampled
    channels of y and of the final state, over the whole sequence."""
    import oracle
    rng = np.random.default_rng(7)
    k = 4 if cfg.L * cfg.N > 1e6 else 16
    chs = sorted({(int(rng.integers(cfg.Bt)), int(rng.integers(cfg.D))) for _ in range(k)} | {(0, 0)})
    bs = np.array([c[0] for c in chs]); ds = np.array([c[1] for c in chs])
    f = gen.as_f64
    rows = lambda t: None if t is None else t[torch.as_tensor(bs), torch.as_tensor(ds), :].to(torch.float64).numpy()  # noqa: E731
    yo, ho, ym, hm = oracle.scan_rows(rows(inp["u"]), rows(inp["delta"]), f(inp["A"])[ds], f(inp["B"]), f(inp["C"]), bs,
                                      D=None if inp["D"] is None else f(inp["D"])[ds], z=rows(inp["z"]),
                                      delta_bias=None if inp["delta_bias"] is None else f(inp["delta_bias"])[ds],
                                      delta_softplus=inp["delta_softplus"], with_mag=True, nthreads=len(chs))
    yg = y[torch.as_tensor(bs), torch.as_tensor(ds), :].float().cpu().double().numpy()
    out = {"channels": [list(c) for c in chs], "y_max_rel_err": float(oracle.rel_err(yg, yo, ym)),
           "tol": 2e-2 if cfg.io == "bf16" else 1e-5,
           "metric": "max |gpu - oracle| / max(|oracle|, magnitude companion), fp64 oracle, whole sequence"}
    if last is not None:
        hg = last[torch.as_tensor(bs), torch.as_tensor(ds), :].cpu().double().numpy()
        out["state_max_rel_err"] = float(oracle.rel_err(hg, ho, hm))
    return out


def bench_config(cfg, dev, stream, timed, ex2_peak, hbm):
    """The forward scan of one workload: ms per call (its own caller workspace), elements/s,
    fraction of the exponential roofline and of HBM bandwidth."""
    from selective_state_space_153_b300 import ssm
    inp = gen.scan_inputs(cfg)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(g["u"])
    last = torch.empty((cfg.Bt, cfg.D, cfg.N), dtype=torch.float32, device=dev) if cfg.last_state else None
    io = ssm.SSM_BF16 if cfg.io == "bf16" else ssm.SSM_F32
    ws_bytes = ssm.workspace_bytes(cfg.Bt, cfg.D, cfg.L, cfg.N, io)
    wsb = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=dev)

    def step():
        ssm.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                               delta_bias=g["delta_bias"], delta_softplus=cfg.softplus, y=y, last_state=last,
                               stream=stream, workspace=wsb)
    ms = timed(step)
    t = ms / 1e3
    return {"workload": config_json(cfg)["workload"], "ms_per_step": ms, "value": cfg.elements / t, "unit": "elem/s",
            "tokens_per_s": cfg.Bt * cfg.L / t, "roofline_frac": cfg.elements / t / 1e9 / ex2_peak,
            "hbm_frac": scan_io_bytes(cfg) / t / 1e9 / hbm,
            "l2": "inputs %.1f MB: %s" % (scan_io_bytes(cfg) / 1e6,
                                          "larger than L2" if scan_io_bytes(cfg) > 126e6 else "L2-resident between calls"),
            "launches_per_step": 3 if ws_bytes > 0 else 1}


def bench_backward(dev, ws, cfg):
    """Gradients of the scan (ssm_selective_scan_bwd), bf16 io with gate and bias, fp32
    gradients: checkpointed forward + reverse adjoint, with the planner's time split where the
    channel blocks alone do not fill the GPU (the batch-8 workload 8 x 1536 x 2048 x 16 runs
    unsplit; 1 x 1536 x 16384 x 16 split)."""
    from selective_state_space_153_b300 import ssm
    inp = gen.scan_inputs(cfg)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dy = torch.randn(g["u"].shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(dev)
    wsb = torch.empty(ssm.load().ssm_selective_scan_bwd_workspace_bytes(
        ctypes_dims(cfg.Bt, cfg.D, cfg.L, cfg.N)), dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()

    def step():
        ssm.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, D=g["D"], z=g["z"],
                               delta_bias=g["delta_bias"], delta_softplus=True, workspace=wsb, stream=s)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    k = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(s)
    for _ in range(k):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws) / k
    # kernels of one call, counted after the timed region (the profiler's hooks stay out of it)
    from torch.profiler import profile, ProfilerActivity
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        step()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type.name == "CUDA" and "bwd" in e.name]
    per_call = len(names)
    elems = cfg.elements
    return {"workload": f"backward of {cfg.name}: Bt={cfg.Bt} D={cfg.D} L={cfg.L} N={cfg.N} bf16 io, fp32 gradients",
            "ms_per_step": ms, "value": ws * elems / (ms / 1e3), "unit": "elem/s",
            "exps_per_element": 3,
            "roofline_frac_of_ex2_peak": 3 * elems / (ms / 1e3) / (SM_COUNT * EX2_PER_CLK_SM * 2032.0e6),
            "kernels_per_call": sorted(set(n.split("(")[0] for n in names)),
            "launches": per_call * (k + 3 + 1)}


def ctypes_dims(Bt, Dm, L, N):
    import ctypes
    from selective_state_space_153_b300 import ssm
    return ctypes.byref(ssm.dims(Bt, Dm, L, N, ssm.SSM_BF16))


def bench_decode(dev):
    """Recurrent step at batch 256 x 5120 channels x 16 states: tok/s = batch / step time,
    L2 flushed before every timed step (the 84 MB state would otherwise stay in L2)."""
    from selective_state_space_153_b300 import ssm
    cfg = gen.DECODE
    d = gen.decode_inputs(cfg)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    st = g["state0"].clone()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    drain = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MB, read after the flush
    ys = torch.empty((cfg.steps, cfg.Bt, cfg.D), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream()

    def one(i):
        ssm.state_update(st, g["x"][i], g["dt"][i], g["A"], g["B"][i], g["C"][i], D=g["D"], z=g["z"][i], y=ys[i],
                         stream=s)
    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    times = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(cfg.steps)]
    for i in range(cfg.steps):
        flush.fill_(i & 0xFF)      # evict the state from L2 ...
        drain.sum()                # ... and write back the flush's dirty lines before timing
        ev[i][0].record(s)
        one(i)
        ev[i][1].record(s)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(cfg.steps):
        one(i)
    e1.record(s)
    torch.cuda.synchronize()
    b2b = e0.elapsed_time(e1) / cfg.steps
    med = statistics.median(times)
    bytes_step = (2 * cfg.Bt * cfg.D * cfg.N * 4 + 4 * cfg.Bt * cfg.D * 2 + 2 * cfg.Bt * cfg.N * 2
                  + cfg.D * cfg.N * 4 + cfg.D * 4)
    peaks, kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    return {"workload": f"decode Bt={cfg.Bt} D={cfg.D} N={cfg.N}, {cfg.steps} successive steps",
            "tok_per_s": cfg.Bt / (med / 1e3), "ms_per_step": med,
            "roofline": {"bound": "hbm", "achieved": bytes_step / (med / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": bytes_step / (med / 1e3) / 1e9 / hbm, "peak_kind": kind,
                         "bytes_per_step": bytes_step,
                         "l2": "flushed before each timed step: 256 MB written, then 256 MB read so that "
                               "no dirty flush data is written back inside the step"},
            "back_to_back_tok_per_s": cfg.Bt / (b2b / 1e3), "launches": 2 * cfg.steps}


# ---------------------------------------------------------------------------- reference arm
def bench_reference(args, rank, ws):
    """The fp64 CPU oracle as it stands, on this host's cores: each step scans a bounded
    sample of the workload's channels over the full sequence."""
    if rank != 0:
        return None
    import oracle
    cfg = workload_config(args)
    inp = gen.scan_inputs(cfg)
    nthreads = os.cpu_count() or 1
    rate1, _, _, t1 = oracle_rate(inp, 0.0, nthreads)   # one channel, to size the sample
    per_ch = t1
    k = int(max(1, min(cfg.Bt * cfg.D, round(2.0 * nthreads / max(per_ch, 1e-6)))))
    f = gen.as_f64
    allch = [(b, d) for b in range(cfg.Bt) for d in range(cfg.D)]
    chs = allch[:: max(1, len(allch) // k)][:k]
    bs = np.array([c[0] for c in chs]); ds = np.array([c[1] for c in chs])
    rows = lambda t: None if t is None else t[torch.as_tensor(bs), torch.as_tensor(ds), :].to(torch.float64).numpy()  # noqa: E731
    a = (rows(inp["u"]), rows(inp["delta"]), f(inp["A"])[ds], f(inp["B"]), f(inp["C"]), bs)
    kw = dict(D=None if inp["D"] is None else f(inp["D"])[ds], z=rows(inp["z"]),
              delta_bias=None if inp["delta_bias"] is None else f(inp["delta_bias"])[ds],
              delta_softplus=inp["delta_softplus"], nthreads=nthreads)
    for _ in range(args.warmup):
        oracle.scan_rows(*a, **kw)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan_rows(*a, **kw)
    el = time.perf_counter() - t
    elems = len(chs) * cfg.L * cfg.N
    v = elems * args.steps / el
    cores = min(nthreads, len(chs))
    sample = f"{len(chs)} of {cfg.Bt * cfg.D} channels per step, full L={cfg.L}, N={cfg.N}, fp64 sequential C"
    return {"impl": "reference", "metric": "scan elements/s (B*D*L*N/s); fraction of the max(HBM, SFU) roofline; decode tok/s",
            "value": v, "unit": "elem/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator, PCG64)",
            "config": config_json(cfg),
            "cpu_baseline": {"value": v, "unit": "elem/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def _spawned_rank(rank, n, port, argv):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(n),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.argv = argv
    main()


def main():
    args = parse()
    if args.measure_ex2:
        if torch.cuda.is_available():
            torch.cuda.set_device(0)
        print(json.dumps({"probe": "ex2.approx.ftz.f32 throughput", "result": probe_ex2(),
                          "unit_rate_per_clk_sm": EX2_PER_CLK_SM}), flush=True)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # no launcher: start the N ranks here, one process per GPU
        import socket
        import torch.multiprocessing as mp
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        mp.spawn(_spawned_rank, args=(args.gpus, port, list(sys.argv)), nprocs=args.gpus, join=True)
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        out = bench_reference(args, rank, ws)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    rank, ws, local = dist_setup(args.gpus)
    out = bench_ours(args, rank, ws, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
