"""The kernels' bounded waits: a wait that runs out is reported, not hidden.

Every data load of the plane kernels completes on an mbarrier whose wait is bounded. Here
the test hook shortens that bound to 1 (a short limit counts SM cycles and is checked
before each probe), so that every wait runs out at once, its copies possibly still in
flight (nothing faults or hangs: every CTA that gives up first waits, with the normal
bound, for the copies it issued, then leaves). The test checks that each kind of call
reports its timeout through wtconv_workspace_status, that backward-weight turns it into NaN
gradients, and that the next ordinary calls on the same workspace are bit-identical to a
clean run and report no timeout.
"""
import numpy as np
import pytest
import torch

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _run(x, dy, p, f, ws, out):
    """forward, backward-data, backward-weight into the tensors of `out`, one workspace."""
    d = B.desc_like(x, p.k, p.levels)
    buf, n = ws
    B.wtconv_forward(d, x, f.w0f, f.b0f, f.wlf, out["y"], buf, n)
    B.wtconv_backward_data(d, dy, f.w0f, f.wlf, out["dx"], buf, n)
    B.wtconv_backward_weight(d, x, dy, p.w0, p.b0, p.s0, p.wl, p.sl, out["dw0"], out["db0"],
                             out["ds0"], out["dwl"], out["dsl"], buf, n)


def test_timed_out_waits_are_reported_and_leave_no_trace():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    wl = WORKLOADS["c4_sweep_bf16"]  # 32 x 128 x 128 x 128, L = 4: many waits per call
    inp = make_inputs(wl)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    desc = B.desc_like(x, p.k, wl.levels)
    f = layer.fold(p, desc)
    nf, nbd, nbw = B.wtconv_workspace_size(desc)
    n = max(nf, nbd, nbw)
    ws = (torch.empty(n, dtype=torch.uint8, device=dev), n)

    def outputs():
        return {"y": torch.empty_like(x), "dx": torch.empty_like(dy),
                "dw0": torch.empty_like(p.w0), "db0": torch.empty_like(p.s0),
                "ds0": torch.empty_like(p.s0), "dwl": torch.empty_like(p.wl),
                "dsl": torch.empty_like(p.sl)}

    clean = outputs()
    _run(x, dy, p, f, ws, clean)
    assert B.wtconv_workspace_status(ws[0]) == 0

    bad = outputs()
    B.wtconv_testing_set_wait_limit_ns(1)
    try:
        _run(x, dy, p, f, ws, bad)
        flags = B.wtconv_workspace_status(ws[0])
    finally:
        B.wtconv_testing_set_wait_limit_ns(0)
    assert flags == 0b111, f"status flags {flags:#05b}: every kind of call must report"
    for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
        assert torch.isnan(bad[name]).all(), name

    again = outputs()
    _run(x, dy, p, f, ws, again)
    assert B.wtconv_workspace_status(ws[0]) == 0
    for name in clean:
        a = clean[name].cpu()
        b = again[name].cpu()
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), name


def test_workspace_status_rejects_null():
    lib = B.load_library()
    flags = B.ctypes.c_int(7)
    assert lib.wtconv_workspace_status(None, None, B.ctypes.byref(flags)) == B.WT_ERR_INVALID_ARG
    assert flags.value == 0
