"""The backward-weight entry point that allocates nothing (wtconv_backward_weight_noalloc).

It exists for callers of this library that cannot provide device memory, e.g. code whose
runtime owns all device memory and forbids raw cudaMalloc, or a latency-critical path that
must not call cudaMalloc because it may synchronize the device. Its scratch is a fixed
4 MiB array inside the library, shared by every call. This test calls it through the C ABI
twice in a row (the second call finds the first call's leftovers in the array) and checks
each result against the ordinary workspace entry point on the same inputs, within the
parameter-gradient tolerance used by the parity tests. This file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import make_inputs, shape_workload
from parity_util import TOL_PARAM, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    # small fp32 case: the whole batch fits in one chunk of the 4 MiB scratch
    (4, 16, 32, 32, 5, 2, "f32"),
    # 256 channels at L = 5: 538 KB of partials per image, so 8 images take two chunks
    (8, 256, 64, 64, 5, 5, "bf16"),
]


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
        g = {name: torch.full_like(t, float("nan")) for name, t in ref.items()}
        B.wtconv_backward_weight_noalloc(desc, x, dy, p.w0, p.b0, p.s0, p.wl, p.sl, g["dw0"],
                                         g["db0"], g["ds0"], g["dwl"], g["dsl"])
        torch.cuda.synchronize()
        for name in ("dw0", "db0", "ds0", "dwl", "dsl"):
            a = g[name].double().cpu().numpy()
            r = ref[name].double().cpu().numpy()
            assert np.isfinite(a).all(), (call, name)
            err = rel_err(a, r)
            assert err <= TOL_PARAM[dtype], (call, name, err)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 1100 channels at k = 5, L = 5 need 2 * 1100 * 526 floats > 4 MiB
    d = B.make_desc(1, 1100, 32, 32, 5, 5, B.WT_F32)
    lib = B.load_library()
    st = lib.wtconv_backward_weight_noalloc(d, 256, 256, 256, None, 256, 256, 256, 256,
                                            None, 256, 256, 256, None)
    assert st == B.WT_ERR_WORKSPACE
