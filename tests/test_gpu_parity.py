"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element,
on the seeded synthetic workloads and on edge shapes. All tests need a GB300."""
import numpy as np
import pytest
import torch

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import WORKLOADS, make_inputs, shape_workload
from parity_util import assert_within, gpu_run, run_and_compare, run_and_compare_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    B.load_library()


def test_c1_small_forward():
    wl = WORKLOADS["c1_small_fwd"]
    errs, _ = run_and_compare(wl)
    assert_within(errs, wl.dtype, wl.name)


@pytest.mark.parametrize("fused", [True, False])
def test_c2_fp32_train(fused):
    wl = WORKLOADS["c2_fp32_train"]
    errs, _ = run_and_compare(wl, fused=fused)
    assert_within(errs, wl.dtype, wl.name)


def test_c2_with_bias_and_base_scale():
    wl = WORKLOADS["c2_fp32_train"]
    errs, _ = run_and_compare(wl, bias_and_scale=True)
    assert_within(errs, wl.dtype, wl.name)


def test_c3_stage1_bf16_full():
    wl = WORKLOADS["c3_stage1_bf16"]
    errs, _ = run_and_compare(wl)
    assert_within(errs, wl.dtype, wl.name)


@pytest.mark.parametrize("levels", [0, 1, 2, 3, 4])
def test_c4_level_sweep_full(levels):
    """The 32x128x128x128 bf16 level sweep (L = 0 is the plain depthwise conv), every
    output element and every parameter gradient against the oracle."""
    wl = WORKLOADS["c4_sweep_bf16"].with_levels(levels)
    errs, _ = run_and_compare_full(wl, chunk=32)
    assert_within(errs, wl.dtype, wl.name)


def test_c5_large_full():
    """The 16x256x256x256 bf16 L = 5 workload (the benchmarked one), every output element
    and every parameter gradient against the oracle."""
    wl = WORKLOADS["c5_large_bf16"]
    errs, _ = run_and_compare_full(wl, chunk=32)
    assert_within(errs, wl.dtype, wl.name)


EDGE = [  # n, c, h, w, k, L, dtype
    (1, 1, 8, 8, 3, 3, "f32"),        # deepest level 1x1
    (2, 3, 48, 40, 5, 3, "f32"),      # ragged deep grids (6x5 at L=3)
    (1, 2, 7, 9, 5, 0, "f32"),        # odd plane, plain depthwise
    (1, 2, 6, 10, 3, 1, "f32"),       # H, W = 2 mod 4
    (2, 2, 136, 72, 5, 3, "bf16"),    # several 64x64 tiles with a ragged tail
    (1, 1, 64, 64, 7, 6, "f32"),      # k = 7 down to a 1x1 level
    (1, 3, 32, 32, 1, 2, "f32"),      # k = 1
    (1, 1, 256, 256, 5, 5, "f32"),    # largest fp32 plane of the workloads
    (3, 5, 20, 12, 5, 2, "bf16"),     # odd channel count, small planes
    (2, 4, 96, 160, 3, 4, "bf16"),    # wide plane, k = 3
]


F16 = [  # fp16 I/O (the pages' half-precision measurements): TMA path and plain path
    (2, 4, 64, 64, 5, 2, "f16"),      # TMA (W * 2 bytes a multiple of 16)
    (2, 3, 40, 36, 5, 2, "f16"),      # W * 2 not a multiple of 16: plain staging
    (1, 2, 128, 96, 7, 4, "f16"),     # k = 7, deep levels
    (2, 2, 56, 56, 3, 3, "f16"),      # stage-1 plane, k = 3
]


ODD = [  # sides that are not multiples of 2^L: carriers zero-padded per level
    (2, 3, 13, 11, 5, 2, "f32"),      # both sides odd, plain staging
    (1, 2, 37, 64, 5, 3, "bf16"),     # odd H on the TMA path (W * 2 bytes % 16 == 0)
    (2, 2, 7, 9, 3, 3, "f32"),        # 7 -> 4 -> 2 -> 1 rows
    (1, 2, 100, 60, 7, 4, "bf16"),    # W * 2 bytes % 16 != 0: plain staging, k = 7
    (1, 1, 5, 5, 5, 5, "f32"),        # more levels than the plane has halvings
    (2, 2, 130, 66, 5, 5, "f16"),     # several tiles with odd carriers at deep levels
]


LARGE = [  # planes whose deep-level state no longer fits in shared memory
    (1, 2, 512, 512, 5, 5, "bf16"),   # the pages' largest sweep plane at L = 5
    (1, 1, 1024, 1024, 3, 5, "f32"),
    (1, 1, 512, 512, 7, 5, "f16"),
    (1, 1, 520, 500, 5, 4, "f32"),    # large and not a multiple of 2^L
]


LAYOUT = [  # the forward's shared-memory layouts (band-pair buffers, where X^(2) lives)
    (1, 2, 192, 128, 7, 4, "f32"),    # one band-pair buffer (a barrier more per tile)
    (1, 1, 256, 256, 7, 5, "bf16"),   # two buffers, X^(2) re-read from the level-2 subbands
    (1, 1, 256, 256, 5, 5, "f32"),    # the same in fp32
    (1, 2, 256, 192, 3, 4, "bf16"),   # level-2 tiles TMA-staged from the slot (2x2 tiles)
    (1, 1, 160, 256, 5, 3, "f16"),    # the same, ragged last tile row
    (1, 2, 150, 136, 5, 3, "bf16"),   # the same on a padded plane (general kernel)
]


GROUP = [  # small deep levels sharing one stage/filter round (stacked in the tiles)
    (1, 2, 256, 256, 5, 8, "f32"),    # forward levels 8..5 in one round; dW 4-5 and 6-8
    (2, 3, 56, 56, 5, 3, "bf16"),     # stage-1 plane: dW levels 2 and 3 together
    (1, 2, 64, 512, 5, 5, "bf16"),    # wide plane: only the last two levels fit a tile
    (1, 1, 2048, 64, 3, 6, "f16"),    # tall plane
    (1, 2, 128, 128, 7, 5, "bf16"),   # k = 7: larger halos, fewer levels per round
    (1, 2, 128, 128, 1, 6, "f32"),    # k = 1: no halo
    (2, 3, 112, 80, 3, 6, "bf16"),    # padded plane (general kernels)
    (1, 2, 128, 96, 5, 4, "f32"),     # forward: level 2 (32x24) alone in a compact round
    (2, 3, 56, 56, 5, 3, "f32"),      # forward: levels 3 and 2 in one round (fp32 gate)
    (2, 2, 40, 72, 3, 4, "f32"),      # forward: levels 4..2 in one round, non-square
]


DEEP = [  # the deepest cascades the boundary accepts (L <= 12)
    (1, 1, 16, 16, 3, 12, "bf16"),    # L = 12: the kernels run on the plane padded to 4096^2
    (1, 2, 40, 24, 5, 10, "f32"),     # L = 10 on a small non-square plane (padded to 1024^2)
    (1, 1, 1024, 1024, 3, 10, "bf16"),  # L = 10 on a whole 1024x1024 plane, down to 1x1
]


@pytest.mark.parametrize("n,c,h,w,k,L,dtype", EDGE + F16 + ODD + LARGE + LAYOUT + GROUP + DEEP)
def test_edge_shapes(n, c, h, w, k, L, dtype):
    wl = shape_workload(n, c, h, w, k, L, dtype, seed=1000 + h + w + k + L)
    errs, _ = run_and_compare(wl, bias_and_scale=True)
    assert_within(errs, wl.dtype, wl.name)


def test_c3_stage1_f16_full():
    """The stage-1 shape with fp16 I/O, every element against the oracle."""
    wl = WORKLOADS["c3_stage1_bf16"].with_dtype("f16")
    errs, _ = run_and_compare_full(wl, chunk=48)
    assert_within(errs, wl.dtype, wl.name)


@pytest.mark.parametrize("wl", [
    WORKLOADS["c3_stage1_bf16"],                           # level-2 sweep: 4 pairs, CTA barriers
    shape_workload(2, 6, 256, 256, 5, 5, "f32", seed=77),  # 2 pairs, per-warp releases
], ids=lambda w: w.name)
def test_backward_is_deterministic(wl):
    inp = make_inputs(wl)
    a = gpu_run(inp, wl.levels, True)
    b = gpu_run(inp, wl.levels, True)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_workspace_errors():
    wl = WORKLOADS["c2_fp32_train"]
    inp = make_inputs(wl)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    desc = B.desc_like(x, p.k, wl.levels)
    _, _, nb = B.wtconv_workspace_size(desc)
    assert nb > 0
    small = torch.empty(nb - 16, dtype=torch.uint8, device=dev)
    g = {k: torch.empty_like(v) for k, v in
         {"dw0": p.w0, "db0": p.s0, "ds0": p.s0, "dwl": p.wl, "dsl": p.sl}.items()}
    with pytest.raises(B.WTConvError) as ei:
        B.wtconv_backward_weight(desc, x, dy, p.w0, p.b0, p.s0, p.wl, p.sl, g["dw0"], g["db0"],
                                 g["ds0"], g["dwl"], g["dsl"], small, small.numel())
    assert ei.value.status == B.WT_ERR_WORKSPACE
    # misaligned input pointer
    with pytest.raises(B.WTConvError) as ei:
        B.wtconv_forward(desc, x.data_ptr() + 4, p.w0, None, p.wl, torch.empty_like(x))
    assert ei.value.status == B.WT_ERR_INVALID_ARG


def _random_case(seed):
    """A seeded random configuration: shape, k, L, I/O dtype (small planes, so that the
    oracle finishes quickly), covering odd sides, rows that TMA can and cannot stage, every
    built k and both one- and multi-tile planes."""
    rng = np.random.default_rng(seed)
    k = int(rng.choice([1, 3, 5, 7]))
    dtype = str(rng.choice(["f32", "bf16", "f16"]))
    h = int(rng.integers(1, 161))
    w = int(rng.integers(1, 161))
    levels = int(rng.integers(0, 7))
    n = int(rng.integers(1, 3))
    c = int(rng.integers(1, 4))
    if rng.random() < 0.5:  # rows of a multiple of 16 bytes: the TMA-staged kernels
        w = max(8, w - w % 8)
    return n, c, h, w, k, levels, dtype


@pytest.mark.parametrize("seed", range(32))
def test_random_shapes(seed):
    n, c, h, w, k, L, dtype = _random_case(seed)
    wl = shape_workload(n, c, h, w, k, L, dtype, seed=5000 + seed)
    errs, _ = run_and_compare(wl, bias_and_scale=True)
    assert_within(errs, wl.dtype, wl.name)


def _random_large_case(seed):
    """Seeded random larger planes: multi-tile level-2 grids and deep states that may move
    to the workspace slot or fall back to one CTA per SM."""
    rng = np.random.default_rng(10_000 + seed)
    k = int(rng.choice([3, 5, 7]))
    dtype = str(rng.choice(["f32", "bf16", "f16"]))
    h = int(rng.integers(130, 601))
    w = int(rng.integers(130, 601))
    if rng.random() < 0.6:
        w -= w % 8
    levels = int(rng.integers(2, 9))
    return 1, 1, h, w, k, levels, dtype


@pytest.mark.parametrize("seed", range(10))
def test_random_large_planes(seed):
    n, c, h, w, k, L, dtype = _random_large_case(seed)
    wl = shape_workload(n, c, h, w, k, L, dtype, seed=6000 + seed)
    errs, _ = run_and_compare(wl, bias_and_scale=True)
    assert_within(errs, wl.dtype, wl.name)
