"""The backward-weight entry point that allocates nothing (wtconv_backward_weight_noalloc).

It exists for callers of this library that cannot provide device memory, e.g. code whose
runtime owns all device memory and forbids raw cudaMalloc, or a latency-critical path that
must not call cudaMalloc because it may synchronize the device. Its scratch is a fixed
4 MiB array inside the library, shared by every call. These tests call it through the C ABI
twice in a row (the second call finds the first call's leftovers in the array) and check
each result against the ordinary workspace entry point on the same inputs, within the
parameter-gradient tolerance used by the parity tests, and once against the oracle; a
forced timeout inside its plane kernel must come back as NaN gradients. This file sorts
last so that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import make_inputs, shape_workload
from parity_util import TOL_PARAM, db0_floor, oracle_run, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    # small fp32 case: the whole batch fits in one chunk of the 4 MiB scratch
    (4, 16, 32, 32, 5, 2, "f32"),
    # 256 channels at L = 5: 526 KB of partials per image, so the 8 images run as four
    # chunks of two
    (8, 256, 64, 64, 5, 5, "bf16"),
    # 128 KB level-2 slots: only 29 fit, fewer than the 64 CTAs the plane kernel would
    # otherwise run, so the grid shrinks and the CTAs take planes from the shared counter
    (2, 64, 256, 256, 5, 5, "bf16"),
    # k = 7 (the one-CTA-per-SM backward-weight kernel) and k = 3 at fp16 I/O
    (4, 24, 96, 96, 7, 3, "bf16"),
    (3, 20, 72, 64, 3, 3, "f16"),
]


def _noalloc(desc, x, dy, p, like):
    g = {name: torch.full_like(t, float("nan")) for name, t in like.items()}
    B.wtconv_backward_weight_noalloc(desc, x, dy, p.w0, p.b0, p.s0, p.wl, p.sl, g["dw0"],
                                     g["db0"], g["ds0"], g["dwl"], g["dsl"])
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("n,c,h,w,k,L,dtype", CASES)
def test_noalloc_matches_workspace_path_on_two_calls(n, c, h, w, k, L, dtype):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    wl = shape_workload(n, c, h, w, k, L, dtype, seed=77 + L)
    inp = make_inputs(wl, bias_and_scale=True)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    ref = layer.backward_weight(x, dy, p)
    desc = B.desc_like(x, p.k, L)
    for call in range(2):
        g = _noalloc(desc, x, dy, p, ref)
        for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
            a = g[name].double().cpu().numpy()
            r = ref[name].double().cpu().numpy()
            assert np.isfinite(a).all(), (call, name)
            err = rel_err(a, r)
            assert err <= TOL_PARAM[dtype], (call, name, err)


def test_noalloc_matches_oracle():
    """The no-alloc gradients against the CPU oracle itself (not only against the workspace
    entry point), on a multi-chunk bf16 case."""
    wl = shape_workload(6, 24, 48, 40, 5, 3, "bf16", seed=91)
    inp = make_inputs(wl, bias_and_scale=True)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    like = {"dw0": p.w0, "db0": p.s0, "ds0": p.s0, "dwl": p.wl, "dsl": p.sl}
    g = _noalloc(B.desc_like(x, p.k, wl.levels), x, dy, p, like)
    ref = oracle_run(inp, wl.levels, True)
    floor = db0_floor(inp)
    for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
        err = rel_err(g[name].double().cpu().numpy(), ref[name],
                      floor if name == "db0" else 0.0)
        assert err <= TOL_PARAM["bf16"], (name, err)


@pytest.mark.parametrize("n,c,h,w,k,L,dtype", [
    (1, 1100, 32, 32, 5, 5, "f32"),    # per-channel terms: 2 x 1100 x 526 floats > 4 MiB
    (1, 1, 2048, 2048, 5, 2, "bf16"),  # spatial term: one level-2 slot of 2 x 1 Mi floats
])
def test_noalloc_rejects_shapes_beyond_its_scratch(n, c, h, w, k, L, dtype):
    """Shapes beyond the documented limit return WT_ERR_WORKSPACE before anything is
    launched. Every argument is a real allocation of its full size, so that even a call
    that were (wrongly) accepted would only touch valid memory."""
    wl = shape_workload(n, c, h, w, k, L, dtype, seed=5)
    inp = make_inputs(wl)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    like = {"dw0": p.w0, "db0": p.s0, "ds0": p.s0, "dwl": p.wl, "dsl": p.sl}
    g = {name: torch.empty_like(t) for name, t in like.items()}
    with pytest.raises(B.WTConvError) as ei:
        B.wtconv_backward_weight_noalloc(B.desc_like(x, k, L), x, dy, p.w0, p.b0, p.s0, p.wl,
                                         p.sl, g["dw0"], g["db0"], g["ds0"], g["dwl"],
                                         g["dsl"])
    assert ei.value.status == B.WT_ERR_WORKSPACE
    torch.cuda.synchronize()


def test_noalloc_reports_a_timed_out_wait_as_nan_gradients():
    """With the kernels' bounded waits shortened to 1 (the test hook; a short limit counts SM
    cycles and is checked before each probe), the plane kernel's waits run out at once; the status word in the fixed array turns
    every gradient into NaN, and the next ordinary call (which clears the word) agrees with
    the workspace path again."""
    wl = shape_workload(8, 32, 128, 128, 5, 4, "bf16", seed=123)
    inp = make_inputs(wl, bias_and_scale=True)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    ref = layer.backward_weight(x, dy, p)
    desc = B.desc_like(x, p.k, wl.levels)
    B.wtconv_testing_set_wait_limit_ns(1)
    try:
        bad = _noalloc(desc, x, dy, p, ref)
    finally:
        B.wtconv_testing_set_wait_limit_ns(0)
    for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
        assert torch.isnan(bad[name]).all(), name
    good = _noalloc(desc, x, dy, p, ref)
    for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
        err = rel_err(good[name].double().cpu().numpy(), ref[name].double().cpu().numpy())
        assert err <= TOL_PARAM["bf16"], (name, err)
