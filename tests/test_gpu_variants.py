"""GPU parity of the staged ablation pipelines (include/wtconv_ablation.h): the reference's
materializing stage chain and each cumulative reformulation against the CPU oracle's
forward, on seeded fp32 inputs covering several tiles, ragged tiles, k in {1, 3, 5, 7}, L
from 0 up to the deepest level a size allows, non-square planes and bias + base scale."""
import pytest
import torch

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300 import layer
from depthwise_receptive_field_gb300.inputs import make_inputs, shape_workload
from parity_util import TOL, oracle_run, rel_err, to64

pytestmark = pytest.mark.gpu

VARIANTS = [B.WT_VARIANT_REFERENCE, B.WT_VARIANT_FUSED_ANALYSIS,
            B.WT_VARIANT_COLLAPSED_SYNTHESIS, B.WT_VARIANT_FOLDED]

SHAPES = [
    # n, c, h, w, k, L
    (2, 3, 64, 64, 5, 2),
    (1, 4, 96, 80, 5, 4),     # ragged 32x64 conv tiles and 32x32 level tiles
    (2, 2, 40, 40, 3, 3),     # deepest level 5x5 (odd plane sides)
    (1, 3, 24, 56, 7, 2),     # non-square
    (2, 2, 32, 32, 1, 5),     # k = 1, deepest level 1x1
    (1, 2, 48, 48, 5, 0),     # no levels: the base path alone
]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: B.VARIANT_NAMES[v])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_variant_matches_oracle(variant, shape):
    n, c, h, w, k, L = shape
    wl = shape_workload(n, c, h, w, k, L, "f32", seed=11 + L, backward=False)
    inp = make_inputs(wl, bias_and_scale=True)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    y = layer.forward_variant(x, p, variant)
    torch.cuda.synchronize()
    ref = oracle_run(inp, L, False)["y"]
    err = rel_err(to64(y), ref)
    assert err <= TOL["f32"], f"{B.VARIANT_NAMES[variant]} {shape}: {err:.3e}"


def test_variants_agree_with_the_fused_forward():
    """All four staged pipelines and the single-pass forward compute the same operator."""
    wl = shape_workload(2, 8, 128, 128, 5, 4, "f32", seed=5, backward=False)
    inp = make_inputs(wl, bias_and_scale=True)
    dev = torch.device("cuda", 0)
    p = layer.Params.from_inputs(inp, dev)
    x = inp["x"].to(dev)
    y_ref = to64(layer.forward(x, p))
    for v in VARIANTS:
        y = to64(layer.forward_variant(x, p, v))
        assert rel_err(y, y_ref) <= TOL["f32"], B.VARIANT_NAMES[v]


def test_variant_rejects_bf16_and_short_workspace():
    d = B.make_desc(1, 2, 32, 32, 5, 2, B.WT_BF16)
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_variant_workspace_size(d, B.WT_VARIANT_REFERENCE)
    assert e.value.status == B.WT_ERR_UNSUPPORTED
    dev = torch.device("cuda", 0)
    d = B.make_desc(1, 2, 32, 32, 5, 2, B.WT_F32)
    nb = B.wtconv_variant_workspace_size(d, B.WT_VARIANT_REFERENCE)
    x = torch.zeros(1, 2, 32, 32, device=dev)
    w0 = torch.zeros(2, 5, 5, device=dev)
    s0 = torch.ones(2, device=dev)
    wl = torch.zeros(2, 2, 4, 5, 5, device=dev)
    sl = torch.ones(2, 2, 4, device=dev)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_forward_variant(d, B.WT_VARIANT_REFERENCE, x, w0, None, s0, wl, sl,
                                 torch.empty_like(x), ws, nb - 256)
    assert e.value.status == B.WT_ERR_WORKSPACE
