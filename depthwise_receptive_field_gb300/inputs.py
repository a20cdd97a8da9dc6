"""Seeded synthetic inputs for the WTConv layer.

This module holds no arithmetic of the method: it only draws random tensors in a fixed,
documented order and rounds them to the I/O dtype. The CUDA path, the oracle, the tests
and the benchmark all take their inputs from here, so both sides see identical bytes.

Recipe (the paper's layer sweep uses synthetic tensors only):
  generation order, one ``torch.Generator('cpu')`` seeded per workload:
    X ~ N(0, 1)            [N, C, H, W]
    dY ~ N(0, 1)           [N, C, H, W]     (only when the workload has a backward pass)
    W^(0) ~ N(0, 0.04)     [C, k, k]        (variance 0.04, i.e. sigma 0.2)
    W^(1..L) ~ N(0, 0.04)  [L, C, 4, k, k]  (one kernel per channel and subband)
    s^(1..L) ~ U(0.05, 0.2) [L, C, 4]
    base scale s^(0) = 1, bias b = 0, unless ``bias_and_scale`` asks for
    s^(0) ~ U(0.5, 1.5) and b ~ N(0, 0.04), drawn after everything above.
  X and dY are drawn in float32 and rounded to bfloat16 or float16 (round to nearest
  even) when the workload's I/O dtype is bf16 or f16; parameters stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    c: int
    h: int
    w: int
    k: int
    levels: int
    dtype: str  # "f32", "bf16" or "f16": the I/O dtype; accumulation is always fp32
    seed: int
    backward: bool

    @property
    def elements(self) -> int:
        return self.n * self.c * self.h * self.w

    @property
    def torch_dtype(self):
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    def with_dtype(self, dtype: str) -> "Workload":
        return replace(self, dtype=dtype, name=f"{self.name}-{dtype}")

    def with_levels(self, levels: int) -> "Workload":
        return replace(self, levels=levels, name=f"{self.name.split('-L')[0]}-L{levels}")


# The five synthetic workloads: a small forward-only case, a mid-size fp32 training case,
# a WTConvNeXt-T stage-1-like layer, a level sweep at 128x128 and a large-spatial stress.
WORKLOADS = {
    "c1_small_fwd": Workload("c1_small_fwd", 1, 8, 32, 32, 5, 1, "f32", 0, False),
    "c2_fp32_train": Workload("c2_fp32_train", 8, 64, 64, 64, 5, 2, "f32", 1, True),
    "c3_stage1_bf16": Workload("c3_stage1_bf16", 64, 96, 56, 56, 5, 3, "bf16", 2, True),
    "c4_sweep_bf16": Workload("c4_sweep_bf16", 32, 128, 128, 128, 5, 4, "bf16", 3, True),
    "c5_large_bf16": Workload("c5_large_bf16", 16, 256, 256, 256, 5, 5, "bf16", 4, True),
}


def make_inputs(wl: Workload, *, bias_and_scale: bool = False, n: int | None = None) -> dict:
    """Draw the workload's tensors on the CPU. Returns a dict of CPU tensors:
    x, dy (I/O dtype; dy is None for forward-only workloads), w0, b0, s0, wl, sl (fp32).
    ``n`` overrides the batch size (the draw order and seed stay the same)."""
    nb = wl.n if n is None else n
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    shape = (nb, wl.c, wl.h, wl.w)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    dy = torch.randn(shape, generator=g, dtype=torch.float32) if wl.backward else None
    w0 = torch.randn((wl.c, wl.k, wl.k), generator=g, dtype=torch.float32) * 0.2
    wlv = torch.randn((wl.levels, wl.c, 4, wl.k, wl.k), generator=g, dtype=torch.float32) * 0.2
    sl = torch.rand((wl.levels, wl.c, 4), generator=g, dtype=torch.float32) * 0.15 + 0.05
    if bias_and_scale:
        s0 = torch.rand((wl.c,), generator=g, dtype=torch.float32) + 0.5
        b0 = torch.randn((wl.c,), generator=g, dtype=torch.float32) * 0.2
    else:
        s0 = torch.ones((wl.c,), dtype=torch.float32)
        b0 = torch.zeros((wl.c,), dtype=torch.float32)
    if wl.dtype in ("bf16", "f16"):
        x = x.to(wl.torch_dtype)
        dy = dy.to(wl.torch_dtype) if dy is not None else None
    return {"x": x, "dy": dy, "w0": w0, "b0": b0, "s0": s0, "wl": wlv, "sl": sl}


# Shape of the pages' measured-traffic table (App. B, Table 11): B = 8, C = 128, H = W = 128,
# k = 5, fp32; used by the ablation of the reformulations (L = 1..5).
ABLATION_SHAPE = (8, 128, 128, 128, 5)


def shape_workload(n, c, h, w, k, levels, dtype="f32", seed=0, backward=True) -> Workload:
    """An ad-hoc workload for edge-case tests (same recipe, any shape)."""
    return Workload(f"shape_{n}x{c}x{h}x{w}_k{k}_L{levels}_{dtype}", n, c, h, w, k, levels,
                    dtype, seed, backward)
