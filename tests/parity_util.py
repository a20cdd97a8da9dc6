"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and the
CPU oracle on the same seeded inputs, and measure their disagreement."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import Workload, make_inputs

# Norm-wise max relative error gates (|gpu - oracle|_max / |oracle|_max): 1e-5 for fp32
# I/O; 2e-2 for bf16 I/O with fp32 accumulation (outputs are rounded to bf16, 2^-9 rel);
# 2e-3 for fp16 I/O (outputs rounded to fp16, 2^-11 rel, with a 4x margin).
TOL = {"f32": 1e-5, "bf16": 2e-2, "f16": 2e-3}
# Parameter gradients are always fp32 sums of products of the (exact) inputs.
TOL_PARAM = {"f32": 1e-5, "bf16": 1e-4, "f16": 1e-4}


def rel_err(got, ref, floor: float = 0.0) -> float:
    """max |got - ref| / max(max |ref|, floor)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = max(float(np.abs(ref).max()), floor)
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


# db0 = s0 * sum(dY) is a plain sum, whose floating-point error is bounded by the sum of the
# absolute terms, not by the sum: a channel whose dY nearly cancels (a single 42x72 plane
# summing to -0.057 out of 2404 in absolute terms) has a tiny reference and an ordinary
# fp32 error of a few 1e-6. Its scale is therefore floored at 1e-3 of s0 * sum|dY| (the
# largest channel's). The fp32 gate then allows an absolute error of 1e-8 * s0 * sum|dY|,
# still below the unit roundoff (6e-8) times that magnitude: an accurately summed result
# is still required.
DB0_FLOOR = 1e-3


def db0_floor(inp: dict, c_idx=None) -> float:
    dy = inp["dy"].to(torch.float64)
    s0 = inp["s0"].to(torch.float64)
    if c_idx is not None:
        ci = torch.as_tensor(c_idx)
        dy, s0 = dy[:, ci], s0[ci]
    mag = (s0.abs() * dy.abs().sum(dim=(0, 2, 3))).max().item()
    return DB0_FLOOR * mag


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def gpu_run(inp: dict, levels: int, backward: bool, fused: bool = True) -> dict:
    """Run fold + forward (+ backward) on cuda:0 through the C ABI."""
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    ws = layer.Workspace(dev)
    desc = layer.B.desc_like(x, p.k, levels)
    f = layer.fold(p, desc)
    out = {"y": layer.forward(x, p, f, ws)}
    if backward:
        dy = inp["dy"].to(dev)
        if fused:
            g = layer.backward(x, dy, p, f, ws)
        else:
            g = layer.backward_weight(x, dy, p, ws)
            g["dx"] = layer.backward_data(dy, p, f, ws)
        out.update(g)
    torch.cuda.synchronize()
    return {k: to64(v) for k, v in out.items()}


def oracle_run(inp: dict, levels: int, backward: bool, n_idx=None, c_idx=None) -> dict:
    """Oracle on the whole input, or on the sub-batch of batch indices n_idx and channels
    c_idx (the layer is independent across planes; parameter gradients of a channel sum
    over the batch, so n_idx must then be the whole batch)."""
    x = inp["x"]
    dy = inp["dy"]
    w0, b0, s0, wl, sl = inp["w0"], inp["b0"], inp["s0"], inp["wl"], inp["sl"]
    if c_idx is not None:
        ci = torch.as_tensor(c_idx)
        x = x[:, ci]
        dy = dy[:, ci] if dy is not None else None
        w0, b0, s0 = w0[ci], b0[ci], s0[ci]
        wl, sl = wl[:, ci], sl[:, ci]
    if n_idx is not None:
        ni = torch.as_tensor(n_idx)
        x = x[ni]
        dy = dy[ni] if dy is not None else None
    out = {"y": oracle.forward(x, w0, b0, s0, wl, sl, levels)}
    if backward:
        g = oracle.backward(x, dy, w0, b0, s0, wl, sl, levels)
        out.update(g)
    return out


def compare(gpu: dict, ref: dict, dtype: str, levels: int, c_idx=None, n_idx=None,
            floors=None) -> dict:
    """Per-tensor relative errors (gpu sliced to the oracle's sub-batch when sampled);
    floors: optional per-tensor lower bounds of the error scale."""
    floors = floors or {}
    errs = {}
    for name, r in ref.items():
        g = gpu[name]
        if name in ("y", "dx"):
            if c_idx is not None:
                g = g[:, list(c_idx)]
            if n_idx is not None:
                g = g[list(n_idx)]
        elif c_idx is not None:
            if name in ("dw0", "db0", "ds0"):
                g = g[list(c_idx)]
            else:
                g = g[:, list(c_idx)]
        if name in ("dwl", "dsl") and levels == 0:
            continue
        errs[name] = rel_err(g, r, floors.get(name, 0.0))
    return errs


def assert_within(errs: dict, dtype: str, what: str = ""):
    for name, e in errs.items():
        tol = TOL[dtype] if name in ("y", "dx") else TOL_PARAM[dtype]
        assert e <= tol, f"{what} {name}: rel err {e:.3e} > {tol:.1e} (all: {errs})"


def run_and_compare(wl: Workload, *, bias_and_scale=False, sample_channels=None, fused=True):
    inp = make_inputs(wl, bias_and_scale=bias_and_scale)
    gpu = gpu_run(inp, wl.levels, wl.backward, fused=fused)
    ref = oracle_run(inp, wl.levels, wl.backward, c_idx=sample_channels)
    floors = {"db0": db0_floor(inp, sample_channels)} if wl.backward else None
    errs = compare(gpu, ref, wl.dtype, wl.levels, c_idx=sample_channels, floors=floors)
    record(wl.name, wl.dtype, errs)
    return errs, gpu


# Achieved errors of the named workload tests, printed as a table at the end of the session
# (tests/conftest.py), so that a loss of precision inside the gates stays visible.
RECORDED: list = []


def record(name: str, dtype: str, errs: dict, abs_errs: dict | None = None):
    RECORDED.append((name, dtype, dict(errs), dict(abs_errs or {})))


def gpu_run_device(inp: dict, levels: int, backward: bool) -> dict:
    """fold + forward (+ the fused backward) on cuda:0 through the C ABI; results stay on
    the device (for comparisons chunk by chunk)."""
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    ws = layer.Workspace(dev)
    desc = layer.B.desc_like(x, p.k, levels)
    f = layer.fold(p, desc)
    out = {"y": layer.forward(x, p, f, ws)}
    if backward:
        out.update(layer.backward(x, inp["dy"].to(dev), p, f, ws))
    torch.cuda.synchronize()
    return out


def run_and_compare_full(wl: Workload, *, chunk: int = 32, bias_and_scale=False):
    """Every output element of the workload against the oracle. The CUDA path runs once on
    the whole tensor; the oracle runs on `chunk` channels at a time (all batch entries, so
    that each channel's parameter gradients are complete), which bounds the host memory.
    Returns the norm-wise relative errors over the whole tensors and the max abs errors."""
    inp = make_inputs(wl, bias_and_scale=bias_and_scale)
    gpu = gpu_run_device(inp, wl.levels, wl.backward)
    diff, mag = {}, {}
    for c0 in range(0, wl.c, chunk):
        ci = list(range(c0, min(wl.c, c0 + chunk)))
        ref = oracle_run(inp, wl.levels, wl.backward, c_idx=ci)
        for name, r in ref.items():
            if name in ("dwl", "dsl") and wl.levels == 0:
                continue
            g = gpu[name]
            g = g[:, c0:c0 + len(ci)] if name in ("y", "dx", "dwl", "dsl") else g[c0:c0 + len(ci)]
            d = float(np.abs(to64(g) - r).max()) if r.size else 0.0
            m = float(np.abs(r).max()) if r.size else 0.0
            diff[name] = max(diff.get(name, 0.0), d)
            mag[name] = max(mag.get(name, 0.0), m)
    floors = {"db0": db0_floor(inp)} if wl.backward else {}
    errs = {}
    for name in diff:
        scale = max(mag[name], floors.get(name, 0.0))
        errs[name] = diff[name] / scale if scale > 0 else diff[name]
    record(wl.name, wl.dtype, errs, diff)
    return errs, diff
