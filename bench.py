#!/usr/bin/env python
"""WTConv layer benchmark on GB300: fwd + bwd throughput (Gelem/s) and roofline fractions.

One step = one pass of the whole layer over one batch:
    fold scales (Eq. 8) -> forward -> backward-data -> backward-weight (+ Eq. 9 unfold)
all through the C ABI of libwtconv, inputs resident in HBM. The default workload is the
largest single-GPU one: N=16, C=256, H=W=256, k=5, L=5, bf16 I/O (X and dY are 537 MB
each, larger than the 126 MB L2, so consecutive steps cannot hit in L2).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak scaling,
no collective on the data path); rank 0 prints one JSON line with the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "WTConv fwd+bwd Gelem/s and achieved HBM GB/s as % of GB300 peak (1 GPU)"
FP32_LANES_PER_SM = 128  # FP32 multiply-add lanes per SM (Blackwell: 4 partitions x 32)
NOMINAL_HBM_GBS = 7900.0
HBM_FALLBACK_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "depthwise_receptive_field_gb300", "csrc")


# ----------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": HBM_FALLBACK_GBS, "source": "fallback"}


def sm_max_mhz(gpu_index: int):
    """The GPU's maximum SM clock as nvidia-smi reports it (None if unavailable)."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={gpu_index}", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        return float(out.splitlines()[0])
    except Exception:
        return None


def derived_fp32_peak_tflops(num_sms: int, mhz: float) -> float:
    """FP32 multiply-add peak from unit counts: SMs x 128 lanes x 2 FLOP x SM clock."""
    return num_sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def measure_fp32_peak(dev, repeats: int = 3) -> dict:
    """Measured FP32 multiply-add throughput: the library's probe kernel (packed f32x2
    multiply-adds on 8 independent chains per thread, 8 CTAs of 256 threads per SM), timed
    with CUDA events on its stream; best of `repeats` runs of ~2 ms each. The scalar form is
    measured beside it."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 20000
    out = torch.empty(blocks * 256, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for packed in (1, 0):
        best = None
        for _ in range(1 + repeats):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            B.wtconv_fma_probe(blocks, iters, packed, out, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)  # first run is a warm-up too
        fmas = blocks * 256 * iters * 8 * (2 if packed else 1)
        res["packed" if packed else "scalar"] = 2 * fmas / (best * 1e-3) / 1e12
    mhz = sm_max_mhz(dev.index or 0)
    return {"tflops": res["packed"], "scalar_tflops": res["scalar"], "num_sms": sms,
            "sm_max_mhz": mhz,
            "derived_tflops": derived_fp32_peak_tflops(sms, mhz) if mhz else None}


def source_sha256() -> str:
    """Hash of the kernel sources' code: line comments, trailing blanks and empty lines are
    left out (the sources have no block comments and no '//' inside strings), so that an
    edit of comments alone keeps a committed ncu summary of the same kernels valid."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name), encoding="utf-8") as f:
                code = [ln.split("//", 1)[0].rstrip() for ln in f]
            h.update(name.encode())
            h.update("\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel sources (its source hash matches); else None."""
    path = os.path.join(PROFILES, f"traffic_{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != source_sha256():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(wl) -> dict:
    return {
        "workload": f"{wl.name}: N={wl.n} C={wl.c} H={wl.h} W={wl.w} k={wl.k} L={wl.levels}, "
                    f"{wl.dtype} I/O, fp32 accumulate",
        "n": wl.n, "c": wl.c, "h": wl.h, "w": wl.w, "k": wl.k, "levels": wl.levels,
        "io_dtype": wl.dtype,
        "step": "fold + forward + backward_data + backward_weight (C ABI)",
        "l2": "no flush: X and dY are each larger than L2, read once per pass",
    }


# ----------------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------------

def oracle_sample(wl, images: int, channels: int):
    """A bounded sample of the workload: `images` batch entries of its first `channels`
    channels, drawn with the workload's recipe and seed at the smaller batch size."""
    from depthwise_receptive_field_gb300.inputs import make_inputs
    inp = make_inputs(wl, n=images)
    sl = slice(0, channels)
    dy = inp["dy"][:, sl] if inp["dy"] is not None else None
    return {"x": inp["x"][:, sl], "dy": dy, "w0": inp["w0"][sl],
            "b0": inp["b0"][sl], "s0": inp["s0"][sl], "wl": inp["wl"][:, sl],
            "sl": inp["sl"][:, sl]}


def time_oracle_step(s: dict, levels: int) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.forward(s["x"], s["w0"], s["b0"], s["s0"], s["wl"], s["sl"], levels)
    if s["dy"] is not None:
        oracle.backward(s["x"], s["dy"], s["w0"], s["b0"], s["s0"], s["wl"], s["sl"], levels)
    return time.perf_counter() - t0


def host_cpu() -> dict:
    """The host's CPU model and logical core count (Linux /proc/cpuinfo)."""
    import platform
    model = None
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip(), val.strip()
                if key == "model name" and model is None:
                    model = val
                elif key in ("CPU implementer", "CPU part") and key not in fields:
                    fields[key] = val
    except OSError:
        pass
    if model is None:
        model = platform.machine() + "".join(f", {k} {v}" for k, v in fields.items())
    return {"cpu_model": model, "os_cpu_count": os.cpu_count()}


def cpu_baseline(wl, target_s: float = 10.0, single_s: float = 3.0, brief: bool = False) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload: up to 8 images of
    all channels on all host cores, passes repeated until about `target_s` seconds of CPU
    work; then one image of up to 64 channels on one thread for about `single_s` seconds
    (the plain-loop figure)."""
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    images = max(1, min(wl.n, 8))
    s = oracle_sample(wl, images, wl.c)
    elems = s["x"].numel()
    total, passes = 0.0, 0
    while total < target_s and passes < 50:
        total += time_oracle_step(s, wl.levels)
        passes += 1
    chans = max(1, min(wl.c, 64))
    s1 = oracle_sample(wl, 1, chans)
    elems1 = s1["x"].numel()
    total1, passes1 = 0.0, 0
    oracle.set_num_threads(1)
    try:
        while total1 < single_s and passes1 < 50:
            total1 += time_oracle_step(s1, wl.levels)
            passes1 += 1
    finally:
        oracle.set_num_threads(cores)
    if brief:
        return {"all_cores_gelem_s": elems * passes / total / 1e9, "cores": cores,
                "one_thread_gelem_s": elems1 * passes1 / total1 / 1e9,
                "sample": f"{images} images x {wl.c} channels on {cores} threads "
                          f"({passes} passes); 1 image x {chans} channels on 1 thread "
                          f"({passes1} passes)"}
    return {"value": elems * passes / total / 1e9, "unit": "Gelem/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{images} of {wl.n} images x all {wl.c} channels ({elems} elements), "
                      f"{passes} fwd+bwd passes in {total:.1f} s, float64 plain loops, "
                      "OpenMP over planes (fwd) and channels (bwd)",
            "single_thread": {
                "value": elems1 * passes1 / total1 / 1e9, "unit": "Gelem/s", "cores": 1,
                "sample": f"1 of {wl.n} images x {chans} of {wl.c} channels ({elems1} "
                          f"elements), {passes1} fwd+bwd passes in {total1:.1f} s"},
            "host": host_cpu()}


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    s = oracle_sample(wl, 1, wl.c)
    elems = s["x"].numel()
    for _ in range(args.warmup):
        time_oracle_step(s, wl.levels)
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle_step(s, wl.levels)
    value = elems * args.steps / total / 1e9
    sample = (f"1 of {wl.n} images x all {wl.c} channels ({elems} elements) per step, "
              "float64 plain loops, OpenMP")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gelem/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "Gelem/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "Gelem/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------------

class Case:
    """One workload's inputs, parameters, outputs and workspace on the device, and its
    training step (fold -> forward -> backward-data -> backward-weight) through the C ABI;
    forward-only workloads stop after the forward."""

    def __init__(self, wl, dev):
        import torch

        from depthwise_receptive_field_gb300 import binding as B
        from depthwise_receptive_field_gb300 import layer
        from depthwise_receptive_field_gb300.inputs import make_inputs

        self.wl = wl
        self.inp = make_inputs(wl)
        self.p = layer.Params.from_inputs(self.inp, dev)
        self.x = self.inp["x"].to(dev)
        self.dy = self.inp["dy"].to(dev) if wl.backward else None
        self.desc = B.desc_like(self.x, self.p.k, wl.levels)
        self.ws = layer.Workspace(dev)
        _, nbd, nbw = B.wtconv_workspace_size(self.desc)
        self.buf, self.bufn = self.ws.get(max(nbd, nbw))
        self.f = layer.fold(self.p, self.desc)
        self.y = torch.empty_like(self.x)
        p = self.p
        self.g = {"dx": torch.empty_like(self.x), "dw0": torch.empty_like(p.w0),
                  "db0": torch.empty_like(p.s0), "ds0": torch.empty_like(p.s0),
                  "dwl": torch.empty_like(p.wl), "dsl": torch.empty_like(p.sl)}
        self.launches = 0

    def step(self, stream, ev=None):
        from depthwise_receptive_field_gb300 import binding as B

        def mark(i):
            if ev is not None:
                ev[i].record(stream)

        p, f, g, d = self.p, self.f, self.g, self.desc
        lv = self.wl.levels > 0
        mark(0)
        B.wtconv_fold_scales(d, p.w0, p.b0, p.s0, p.wl if lv else None, p.sl if lv else None,
                             f.w0f, f.b0f, f.wlf if lv else None, stream)
        self.launches += B.wtconv_last_launch_count()
        mark(1)
        B.wtconv_forward(d, self.x, f.w0f, f.b0f, f.wlf if lv else None, self.y, self.buf,
                         self.bufn, stream)
        self.launches += B.wtconv_last_launch_count()
        mark(2)
        if self.wl.backward:
            B.wtconv_backward_data(d, self.dy, f.w0f, f.wlf if lv else None, g["dx"], self.buf,
                                   self.bufn, stream)
            self.launches += B.wtconv_last_launch_count()
        mark(3)
        if self.wl.backward:
            B.wtconv_backward_weight(d, self.x, self.dy, p.w0, p.b0, p.s0,
                                     p.wl if lv else None, p.sl if lv else None, g["dw0"],
                                     g["db0"], g["ds0"], g["dwl"] if lv else None,
                                     g["dsl"] if lv else None, self.buf, self.bufn, stream)
            self.launches += B.wtconv_last_launch_count()
        mark(4)


def segments(evs) -> dict:
    """Mean per-pass milliseconds from the per-step event quintuples."""
    seg = {"fold": 0.0, "forward": 0.0, "backward_data": 0.0, "backward_weight": 0.0}
    for ev in evs:
        seg["fold"] += ev[0].elapsed_time(ev[1])
        seg["forward"] += ev[1].elapsed_time(ev[2])
        seg["backward_data"] += ev[2].elapsed_time(ev[3])
        seg["backward_weight"] += ev[3].elapsed_time(ev[4])
    return {k: v / len(evs) for k, v in seg.items()}


def roofs(wl, seg_ms: dict, step_ms: float, peak_tf: float, hbm_gbs: float) -> dict:
    """FP32-ALU fraction of the dominant plane kernel and HBM fraction of the step's ideal
    bytes, from per-pass times."""
    from depthwise_receptive_field_gb300 import iomodel
    alg = iomodel.algorithmic(wl.k, wl.levels, 4 if wl.dtype == "f32" else 2)
    if wl.backward:
        fwd_ms = (seg_ms["forward"] + seg_ms["backward_data"]) / 2
        dw_ms = seg_ms["backward_weight"]
        if 2 * fwd_ms >= dw_ms:
            dom, dom_ms, dom_alg = "wt_fwd_plane_kernel", fwd_ms, alg["forward"]
        else:
            dom, dom_ms, dom_alg = "wt_dw_plane_kernel", dw_ms, alg["backward_weight"]
        step_bytes = wl.elements * sum(a["bytes"] for a in alg.values())
    else:
        dom, dom_ms, dom_alg = "wt_fwd_plane_kernel", seg_ms["forward"], alg["forward"]
        step_bytes = wl.elements * alg["forward"]["bytes"]
    tflops = wl.elements * dom_alg["flops"] / (dom_ms * 1e-3) / 1e12
    gbs = step_bytes / (step_ms * 1e-3) / 1e9
    return {"kernel": dom, "kernel_ms": dom_ms, "achieved_tflops": tflops,
            "alu_frac": tflops / peak_tf, "flops_per_element": dom_alg["flops"],
            "step_bytes": step_bytes, "hbm_gbs": gbs, "hbm_frac": gbs / hbm_gbs}


def run_per_config(args, dev, stream, peak_tf: float, hbm_gbs: float, with_oracle: bool):
    """Every other synthetic workload (the small forward-only case, the fp32 and stage-1
    training cases, the 128x128 level sweep at L = 0..4), timed as the pages' layer
    benchmark does (20 warm-up and 50 timed steps, WTConv-IO §5.1) with L2 flushed before
    every timed step (these inputs are near or below the L2 size), each with the oracle
    timed on a bounded sample on all host cores and on one thread."""
    import torch

    from depthwise_receptive_field_gb300.inputs import WORKLOADS
    wls = [WORKLOADS["c1_small_fwd"], WORKLOADS["c2_fp32_train"], WORKLOADS["c3_stage1_bf16"]]
    wls += [WORKLOADS["c4_sweep_bf16"].with_levels(L) for L in range(5)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = []
    for wl in wls:
        case = Case(wl, dev)
        for _ in range(20):
            case.step(stream)
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(50)]
        for ev in evs:
            flush.fill_(1)
            case.step(stream, ev)
        torch.cuda.synchronize()
        seg = segments(evs)
        step_ms = sum(seg.values())
        passes = 3 if wl.backward else 1
        entry = {"workload": workload_config(wl)["workload"],
                 "gelem_s": wl.elements / (step_ms * 1e-3) / 1e9,
                 "ms_per_step": step_ms, "segments_ms": seg,
                 "passes": "fold + forward + backward_data + backward_weight" if passes == 3
                 else "fold + forward", "steps": 50, "warmup": 20,
                 "l2": "flushed (256 MB write) before every timed step"}
        entry.update(roofs(wl, seg, step_ms, peak_tf, hbm_gbs))
        if with_oracle:
            entry["oracle"] = cpu_baseline(wl, target_s=1.5, single_s=0.7, brief=True)
        out.append(entry)
        del case
        torch.cuda.empty_cache()
    return out


def run_noalloc(case, stream, steps: int = 5) -> dict:
    """The backward-weight entry point without a workspace on the same workload (its
    fixed 4 MiB scratch bounds its grid on large planes), timed beside the workspace path."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    p, g, lv = case.p, case.g, case.wl.levels > 0

    def call():
        B.wtconv_backward_weight_noalloc(case.desc, case.x, case.dy, p.w0, p.b0, p.s0,
                                         p.wl if lv else None, p.sl if lv else None, g["dw0"],
                                         g["db0"], g["ds0"], g["dwl"] if lv else None,
                                         g["dsl"] if lv else None, stream)
    try:
        call()
    except Exception as e:  # e.g. a shape beyond the 4 MiB scratch
        return {"unavailable": str(e)}
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return {"ms": e0.elapsed_time(e1) / steps, "steps": steps}


def run_ours(args, wl):
    import torch

    from depthwise_receptive_field_gb300 import binding as B

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    B.load_library()
    stream = torch.cuda.current_stream(dev)
    peaks = measured_peaks()

    case = Case(wl, dev)
    # the end-to-end figure first, before any other GPU work of this process: taken after
    # the device-resident timing it came out at about twice its copy bound on the GB300
    # machines measured, taken first it runs at the bound (the step's copies are the
    # bottleneck, not the kernels)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, case.inp, case.p, case.f, case.desc, case.buf, case.bufn,
                      stream, world, dev)
    fp32 = measure_fp32_peak(dev)
    peak_tf = fp32["tflops"]
    for _ in range(max(3, args.warmup)):
        case.step(stream)
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    case.launches = 0
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        case.step(stream, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, dev)
    seg_ms = segments(evs)

    elems = wl.elements
    value = world * elems * args.steps / (total_ms * 1e-3) / 1e9
    rf = roofs(wl, seg_ms, total_ms / args.steps, peak_tf, peaks["hbm_gbs"])
    traffic = committed_traffic(rf["kernel"], wl.name)

    result = {
        "metric": METRIC, "value": value, "unit": "Gelem/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl),
        "roofline": {
            "bound": "alu", "kernel": rf["kernel"], "achieved": rf["achieved_tflops"],
            "peak": peak_tf, "unit": "TFLOP/s", "frac": rf["achieved_tflops"] / peak_tf,
            "traffic": traffic,
            "peak_source": "measured: FP32 multiply-add probe (packed f32x2, "
                           f"{fp32['num_sms']} SMs x 8 CTAs x 256 threads, best of 3)",
            "derived_peak": fp32["derived_tflops"],
            "derived_peak_source": f"{fp32['num_sms']} SMs (queried) x {FP32_LANES_PER_SM} "
                                   f"FP32 lanes x 2 FLOP x {fp32['sm_max_mhz']} MHz "
                                   "(nvidia-smi clocks.max.sm)",
            "scalar_fma_tflops": fp32["scalar_tflops"],
            "algorithmic_flops_per_element": rf["flops_per_element"],
            "kernel_ms": rf["kernel_ms"],
        },
        "hbm": {
            "achieved_gbs": rf["hbm_gbs"], "peak_gbs": peaks["hbm_gbs"],
            "frac": rf["hbm_frac"], "peak_source": peaks["source"],
            "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": rf["hbm_gbs"] / NOMINAL_HBM_GBS,
            "nominal_source": "nominal HBM3e bandwidth of one GB300 GPU (7.9 TB/s)",
            "algorithmic_bytes_per_step": rf["step_bytes"],
        },
        "segments_ms": seg_ms,
        "clocks": clk,
        "gpu_launches": case.launches,
    }

    if wl.levels > 0 and not args.no_depthwise:
        result["depthwise_context"] = run_depthwise_context(args, wl, case.p, case.x, case.dy,
                                                            case.g, stream, dev, peak_tf)
    if e2e is not None:
        result["e2e"] = e2e
    if not args.no_noalloc:
        result["noalloc_backward_weight"] = dict(
            run_noalloc(case, stream), workspace_path_ms=seg_ms["backward_weight"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
    if not args.no_per_config:
        del case
        torch.cuda.empty_cache()
        result["per_config"] = run_per_config(args, dev, stream, peak_tf, peaks["hbm_gbs"],
                                              with_oracle=(rank == 0 and world == 1
                                                           and not args.no_cpu_baseline))
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_depthwise_context(args, wl, p, x, dy, g, stream, dev, peak_tf) -> dict:
    """The same-shape plain depthwise k x k conv (this layer at L = 0: base conv + bias and
    scale, no wavelet levels), forward + backward-data + backward-weight through the same
    C ABI, timed like the main step. Context for what the wavelet levels cost on top."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    from depthwise_receptive_field_gb300 import iomodel, layer

    desc0 = B.desc_like(x, p.k, 0)
    _, nbd, nbw = B.wtconv_workspace_size(desc0)
    ws0 = layer.Workspace(dev)
    buf0, bufn0 = ws0.get(max(nbd, nbw))
    w0f = torch.empty_like(p.w0)
    b0f = torch.empty_like(p.s0)
    y0 = torch.empty_like(x)
    steps = max(5, min(args.steps, 50))

    def step():
        B.wtconv_fold_scales(desc0, p.w0, p.b0, p.s0, None, None, w0f, b0f, None, stream)
        B.wtconv_forward(desc0, x, w0f, b0f, None, y0, buf0, bufn0, stream)
        B.wtconv_backward_data(desc0, dy, w0f, None, g["dx"], buf0, bufn0, stream)
        B.wtconv_backward_weight(desc0, x, dy, p.w0, p.b0, p.s0, None, None, g["dw0"],
                                 g["db0"], g["ds0"], None, None, buf0, bufn0, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    alg = iomodel.algorithmic(wl.k, 0, 4 if wl.dtype == "f32" else 2)
    flops = wl.elements * sum(a["flops"] for a in alg.values())
    return {"op": f"plain depthwise {wl.k}x{wl.k} conv, same shape (this library at L=0)",
            "value": wl.elements / (ms * 1e-3) / 1e9, "unit": "Gelem/s", "ms_per_step": ms,
            "steps": steps, "alu_tflops": flops / (ms * 1e-3) / 1e12,
            "alu_frac": flops / (ms * 1e-3) / 1e12 / peak_tf}


def run_ablation(args) -> int:
    """The cumulative ablation of the reformulations (forward pass, fp32): the reference's
    materializing stage chain, + fused analysis, + collapsed synthesis, + folded scales (the
    pages' fused plan), and this library's single-pass forward, on the 8 x 128 x 128 x 128,
    k = 5 shape of the pages' traffic table, for L = 1..5 (or --levels). One JSON line per
    (L, variant): device time per forward (L2 flushed before every timed call), Gelem/s,
    speedup over the reference, and the modeled HBM traffic of the variant.
    With --nvtx, one extra call per (L, variant) runs inside an NVTX push/pop range named
    "wt_measured" (for a counter capture restricted to those calls; each line's "launches"
    says how many kernels of the capture belong to it, in the printed order)."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    from depthwise_receptive_field_gb300 import iomodel, layer
    from depthwise_receptive_field_gb300.inputs import ABLATION_SHAPE, make_inputs, shape_workload

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.load_library()
    n, c, h, w, k = ABLATION_SHAPE
    if args.ablation_n is not None:
        n = args.ablation_n
    levels = [args.levels] if args.levels is not None else [1, 2, 3, 4, 5]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > L2
    stream = torch.cuda.current_stream(dev)
    names = dict(B.VARIANT_NAMES)
    names[-1] = "single_pass"
    for L in levels:
        wl = shape_workload(n, c, h, w, k, L, "f32", seed=7, backward=False)
        inp = make_inputs(wl, bias_and_scale=True)
        p = layer.Params.from_inputs(inp, dev)
        x = inp["x"].to(dev)
        y = torch.empty_like(x)
        ws = layer.Workspace(dev)
        desc = B.desc_like(x, k, L)

        def call(v):
            if v < 0:  # scale fold + the single-pass forward
                layer.forward(x, p, layer.fold(p, desc), ws, y)
            else:
                layer.forward_variant(x, p, v, ws, y)

        times, launches = {}, {}
        for v in (0, 1, 2, 3, -1):
            for _ in range(max(3, args.warmup)):
                call(v)
            launches[v] = B.wtconv_last_launch_count() + (1 if v < 0 else 0)  # + the fold
            tot = 0.0
            for _ in range(args.steps):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(v)
                e1.record(stream)
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            times[v] = tot / args.steps
            if args.nvtx:
                flush.fill_(1)
                torch.cuda.synchronize()
                torch.cuda.nvtx.range_push("wt_measured")
                call(v)
                torch.cuda.nvtx.range_pop()
                torch.cuda.synchronize()
        for v in (0, 1, 2, 3, -1):
            q = iomodel.q_variant(v, L) if v >= 0 else 2.0
            ms = times[v]
            print(json.dumps({
                "ablation": names[v], "levels": L, "shape": [n, c, h, w], "k": k,
                "dtype": "f32", "ms": ms, "gelem_s": wl.elements / (ms * 1e-3) / 1e9,
                "speedup_vs_reference": times[0] / ms,
                "model_traffic_per_element": q,
                "model_gbs": q * wl.elements * 4 / (ms * 1e-3) / 1e9,
                "steps": args.steps, "l2": "flushed (256 MB write) before every timed call",
                "launches": launches[v],
            }), flush=True)
    return 0


PHASES_FWD = {0: "plane setup", 1: "level-2 sweep and weights", 2: "carriers",
              3: "grouped small levels", 4: "level >= 3 stage", 5: "level >= 3 filter, barriers",
              6: "level-2 tile wait and repack (or stage)", 7: "cascade of levels >= 4 into Z^(3)",
              8: "level-2 barrier", 9: "level-2 filter", 10: "level-2 deep sums, barrier",
              11: "end of deep phase", 12: "full-resolution remainder", 13: "plane end",
              14: "tile wait", 15: "band conversion", 16: "barrier A, next tile issued",
              17: "level-1 filter", 18: "base filter, synthesis, store"}
PHASES_DW = {0: "plane setup", 1: "level-2 sweep", 3: "tile pair wait",
             4: "band conversions, dY sum", 5: "barrier B1, next pair issued",
             6: "correlations (base | level 1)", 7: "barrier B2", 8: "flush, partial vector",
             9: "plane end", 10: "grouped small levels", 11: "tiled level stage",
             12: "tiled level barrier 1", 13: "tiled level correlations",
             14: "tiled level barrier 2", 15: "tiled level flush"}


def run_phase_clocks(args, wl) -> int:
    """Per-phase clocks of the two plane kernels on one workload: builds the library with the
    clocks compiled in (a separate build; the ordinary library has none of that code), runs
    `warmup` + `steps` forward and backward-weight calls, and prints, per kernel, the cycles
    thread 0 of a CTA spends in each phase per plane and their shares. With two CTAs per SM
    each CTA is timed while the other runs: the shares say where a CTA's time goes, not what
    a phase would cost alone. The clocks add a little time; no bench figure comes from this
    mode."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    from depthwise_receptive_field_gb300 import build as _build
    from depthwise_receptive_field_gb300 import layer
    from depthwise_receptive_field_gb300.inputs import make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    B.use_library(_build.build_phase_clocks())
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = make_inputs(wl)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    p = layer.Params.from_inputs(inp, dev)
    desc = B.desc_like(x, p.k, wl.levels)
    f = layer.fold(p, desc)
    ws = layer.Workspace(dev)
    y = torch.empty_like(x)
    steps = max(1, min(args.steps, 20))
    for _ in range(max(1, args.warmup)):
        layer.forward(x, p, f, ws, y)
        layer.backward_weight(x, dy, p, ws)
    torch.cuda.synchronize()
    B.wtconv_debug_phase_clocks(0, reset=True)
    B.wtconv_debug_phase_clocks(1, reset=True)
    for _ in range(steps):
        layer.forward(x, p, f, ws, y)
        layer.backward_weight(x, dy, p, ws)
    torch.cuda.synchronize()
    out = {"mode": "phase_clocks", "workload": wl.name, "steps": steps, "kernels": {}}
    for kern, names in ((0, PHASES_FWD), (1, PHASES_DW)):
        v = B.wtconv_debug_phase_clocks(kern)
        planes = v[31]
        total = sum(v[:31])
        rows = {names.get(i, f"phase {i}"): {"cycles_per_plane": v[i] / max(planes, 1),
                                             "share": v[i] / max(total, 1)}
                for i in range(31) if v[i]}
        name = "wt_fwd_plane_kernel" if kern == 0 else "wt_dw_plane_kernel"
        out["kernels"][name] = {"planes": planes, "cycles_per_plane": total / max(planes, 1),
                                "phases": rows}
        print(f"{name}: {planes} planes, {total / max(planes, 1):.0f} cycles per plane (thread 0)")
        for k, r in rows.items():
            print(f"  {k:40s} {r['cycles_per_plane']:9.0f}  {100 * r['share']:5.1f}%")
    print(json.dumps(out))
    return 0


def run_memory(args, wl) -> int:
    """Peak device memory of one training step (fold + forward + backward-data +
    backward-weight through the C ABI), from a clean allocator state: the input X, the
    incoming gradient dY, parameters, outputs, gradients and workspace. Reported for the
    wavelet layer, for the same-shape plain depthwise conv (L = 0), and, for fp32 I/O, for
    the forward of the reference's materializing stage chain (its intermediates are what a
    framework keeps for the backward pass, so this is a lower bound on its training peak).
    Units: bytes and multiples of the input tensor's size (the analogue of the pages'
    Tables 4, 5 and 9)."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B
    from depthwise_receptive_field_gb300 import layer
    from depthwise_receptive_field_gb300.inputs import make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.load_library()
    inp = make_inputs(wl)
    x_bytes = wl.elements * (4 if wl.dtype == "f32" else 2)

    def measure(levels: int, staged_reference: bool = False) -> int:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        p = layer.Params.from_inputs(inp, dev)
        if levels == 0:
            p = layer.Params(p.w0, p.b0, p.s0, p.wl[:0], p.sl[:0])
        x = inp["x"].to(dev)
        if staged_reference:
            y = layer.forward_variant(x, p, B.WT_VARIANT_REFERENCE)
        else:
            dy = inp["dy"].to(dev)
            ws = layer.Workspace(dev)
            f = layer.fold(p, B.desc_like(x, p.k, levels))
            y = layer.forward(x, p, f, ws)
            g = layer.backward(x, dy, p, f, ws)
            del g, dy, ws, f
        torch.cuda.synchronize()
        peak = torch.cuda.max_memory_allocated(dev) - base
        del y, x, p
        return peak

    out = {"memory": True, "workload": workload_config(wl)["workload"],
           "input_bytes": x_bytes}
    peak = measure(wl.levels)
    dw = measure(0)
    out["wtconv_step_peak_bytes"] = peak
    out["wtconv_step_peak_x_input"] = peak / x_bytes
    out["depthwise_step_peak_bytes"] = dw
    out["depthwise_step_peak_x_input"] = dw / x_bytes
    out["wtconv_over_depthwise"] = peak / dw
    if wl.dtype == "f32" and wl.levels > 0:
        ref = measure(wl.levels, staged_reference=True)
        out["reference_forward_peak_bytes"] = ref
        out["reference_forward_peak_x_input"] = ref / x_bytes
        out["wtconv_step_over_reference_forward"] = peak / ref
    else:
        out["reference_forward_peak_bytes"] = None
        out["reference_note"] = "the staged reference pipeline is fp32-only"
    print(json.dumps(out), flush=True)
    return 0


def run_e2e(args, wl, inp, p, f, desc, buf, bufn, stream, world, dev) -> dict:
    """Same step through the public API, with every step's inputs copied from pinned host
    memory and its results (Y, dX and all parameter gradients) copied back, inside the
    timed region. Copies run on their own streams and overlap the neighbouring steps'
    compute (two device buffer sets); each step still moves all of its own bytes."""
    import torch

    from depthwise_receptive_field_gb300 import binding as B

    lv = wl.levels > 0
    xh = inp["x"].pin_memory()
    dyh = inp["dy"].pin_memory()
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    s_cmp = stream

    def dev_set():
        return {"x": torch.empty_like(xh, device=dev), "dy": torch.empty_like(dyh, device=dev),
                "y": torch.empty_like(xh, device=dev), "dx": torch.empty_like(dyh, device=dev),
                "dw0": torch.empty_like(p.w0), "db0": torch.empty_like(p.s0),
                "ds0": torch.empty_like(p.s0), "dwl": torch.empty_like(p.wl),
                "dsl": torch.empty_like(p.sl)}

    def host_set(d):
        return {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                for k, v in d.items() if k not in ("x", "dy")}

    sets = [dev_set(), dev_set()]
    hosts = [host_set(sets[0]), host_set(sets[1])]
    wsb = [buf, torch.empty(bufn, dtype=torch.uint8, device=dev) if bufn else None]
    h2d = xh.numel() * xh.element_size() + dyh.numel() * dyh.element_size()
    d2h = sum(v.numel() * v.element_size() for v in hosts[0].values())
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("h2d", "cmp", "d2h")}
    for k in ev:
        for e in ev[k]:
            e.record(s_cmp)

    def step(i):
        j = i & 1
        d, h = sets[j], hosts[j]
        s_h2d.wait_event(ev["cmp"][j])  # the previous use of this set is computed
        with torch.cuda.stream(s_h2d):
            d["x"].copy_(xh, non_blocking=True)
            d["dy"].copy_(dyh, non_blocking=True)
        ev["h2d"][j].record(s_h2d)
        s_cmp.wait_event(ev["h2d"][j])
        s_cmp.wait_event(ev["d2h"][j])  # its results from two steps ago have left
        B.wtconv_fold_scales(desc, p.w0, p.b0, p.s0, p.wl if lv else None,
                             p.sl if lv else None, f.w0f, f.b0f, f.wlf if lv else None, s_cmp)
        B.wtconv_forward(desc, d["x"], f.w0f, f.b0f, f.wlf if lv else None, d["y"], wsb[j],
                         bufn, s_cmp)
        B.wtconv_backward(desc, d["x"], d["dy"], f.w0f, f.wlf if lv else None, p.w0, p.b0,
                          p.s0, p.wl if lv else None, p.sl if lv else None, d["dx"], d["dw0"],
                          d["db0"], d["ds0"], d["dwl"] if lv else None,
                          d["dsl"] if lv else None, wsb[j], bufn, s_cmp)
        ev["cmp"][j].record(s_cmp)
        s_d2h.wait_event(ev["cmp"][j])
        with torch.cuda.stream(s_d2h):
            for k in h:
                h[k].copy_(d[k], non_blocking=True)
        ev["d2h"][j].record(s_d2h)

    # Five blocks of up to 20 steps each, the median block reported and every block listed:
    # on the shared GB300 hosts single blocks intermittently take up to twice the copy
    # bound (the two copy directions then stop overlapping) while the link probe right
    # after is unchanged, so one block alone is a noisy figure.
    steps = max(2, min(args.steps, 20))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    blocks = []
    for _ in range(5):
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_h2d)
        for i in range(steps):
            step(i)
        b.record(s_d2h)
        torch.cuda.synchronize()
        blocks.append(max_over_ranks(a.elapsed_time(b), world, dev) / steps)
    ms_step = sorted(blocks)[len(blocks) // 2]
    link = host_link(xh, sets[0]["x"], hosts[0]["y"], sets[0]["y"], s_h2d, s_d2h)
    bound_ms = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                   (h2d + d2h) / (link["both_gbs"] * 1e9)) * 1e3
    return {"value": world * wl.elements / (ms_step * 1e-3) / 1e9, "unit": "Gelem/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms_step,
            "blocks_ms_per_step": blocks,
            "timing": f"median of {len(blocks)} blocks of {steps} steps",
            "pipeline": "H2D, compute and D2H on separate streams; two device buffer sets",
            "host_link": link, "copy_bound_ms_per_step": bound_ms}


def host_link(h_src, d_dst, h_dst, d_src, s_h2d, s_d2h, repeats: int = 3) -> dict:
    """Pinned host <-> device copy bandwidth of this machine (best of `repeats`), each direction
    alone and both at once: the bound on the end-to-end figure."""
    import torch

    def timed(fn):
        best = None
        for _ in range(repeats):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return best

    def h2d():
        with torch.cuda.stream(s_h2d):
            d_dst.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_d2h):
            h_dst.copy_(d_src, non_blocking=True)

    def both():
        h2d()
        d2h()

    nb_h = h_src.numel() * h_src.element_size()
    nb_d = d_src.numel() * d_src.element_size()
    return {"h2d_gbs": nb_h / timed(h2d) / 1e9, "d2h_gbs": nb_d / timed(d2h) / 1e9,
            "both_gbs": (nb_h + nb_d) / timed(both) / 1e9}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5_large_bf16")
    ap.add_argument("--levels", type=int, default=None,
                    help="override the workload's L (e.g. the 128x128 level sweep)")
    ap.add_argument("--io", choices=["f32", "bf16", "f16"], default=None,
                    help="override the workload's I/O dtype (the pages also measure fp16)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ablation", action="store_true",
                    help="time the staged ablation pipelines instead of the training step")
    ap.add_argument("--memory", action="store_true",
                    help="report the peak device memory of one training step instead")
    ap.add_argument("--ablation-n", type=int, default=None,
                    help="with --ablation: batch size (default 8, the pages' traffic table)")
    ap.add_argument("--nvtx", action="store_true",
                    help="with --ablation: one extra call per variant inside an NVTX range")
    ap.add_argument("--no-depthwise", action="store_true",
                    help="skip the same-shape plain depthwise conv context line")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' per-config figures")
    ap.add_argument("--no-noalloc", action="store_true",
                    help="skip timing the no-workspace backward-weight entry point")
    ap.add_argument("--phase-clocks", action="store_true",
                    help="print the plane kernels' per-phase clocks instead (separate build)")
    args = ap.parse_args(argv)
    if args.ablation:
        return run_ablation(args)

    from depthwise_receptive_field_gb300.inputs import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.levels is not None:
        wl = wl.with_levels(args.levels)
    if args.io is not None and args.io != wl.dtype:
        wl = wl.with_dtype(args.io)
    if not wl.backward:
        raise SystemExit(f"{wl.name} is forward-only; the benchmarked step needs dY")
    if args.memory:
        return run_memory(args, wl)
    if args.phase_clocks:
        return run_phase_clocks(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
