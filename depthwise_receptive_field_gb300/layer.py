"""WTConv layer on top of the C ABI: torch supplies device memory and streams only.

Every step of the computation runs in libwtconv's CUDA kernels; this module allocates
outputs and the workspace with torch and calls the entry points in order.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class Params:
    """Unfolded parameters (device fp32): w0 [C,k,k], b0 [C], s0 [C], wl [L,C,4,k,k], sl [L,C,4]."""
    w0: torch.Tensor
    b0: torch.Tensor | None
    s0: torch.Tensor
    wl: torch.Tensor
    sl: torch.Tensor

    @property
    def k(self) -> int:
        return int(self.w0.shape[-1])

    @property
    def levels(self) -> int:
        return int(self.wl.shape[0])

    @staticmethod
    def from_inputs(inp: dict, device="cuda") -> "Params":
        def dev(t):
            return None if t is None else t.to(device=device, dtype=torch.float32).contiguous()
        wl = inp["wl"]
        sl = inp["sl"]
        return Params(dev(inp["w0"]), dev(inp["b0"]), dev(inp["s0"]), dev(wl), dev(sl))


@dataclass
class Folded:
    w0f: torch.Tensor
    b0f: torch.Tensor
    wlf: torch.Tensor


def _empty_level_tensor(p: Params, like: torch.Tensor) -> torch.Tensor:
    return torch.empty_like(like) if like.numel() else like


def fold(p: Params, desc: B.wt_desc, stream=None) -> Folded:
    w0f = torch.empty_like(p.w0)
    b0f = torch.empty_like(p.s0)
    wlf = torch.empty_like(p.wl)
    B.wtconv_fold_scales(desc, p.w0, p.b0, p.s0, p.wl if p.levels else None,
                         p.sl if p.levels else None, w0f, b0f, wlf if p.levels else None,
                         stream)
    return Folded(w0f, b0f, wlf)


class Workspace:
    """A reusable device workspace, grown on demand (torch allocator)."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()


def forward(x: torch.Tensor, p: Params, f: Folded | None = None, ws: Workspace | None = None,
            y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    desc = B.desc_like(x, p.k, p.levels)
    f = f or fold(p, desc, stream)
    y = torch.empty_like(x) if y is None else y
    nb, _, _ = B.wtconv_workspace_size(desc)
    buf, size = (ws or Workspace(x.device)).get(nb)
    B.wtconv_forward(desc, x, f.w0f, f.b0f, f.wlf if p.levels else None, y, buf, size, stream)
    return y


def forward_variant(x: torch.Tensor, p: Params, variant: int, ws: Workspace | None = None,
                    y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The forward computed by one of the staged ablation pipelines (fp32 only): the
    reference's materializing stages or one of its cumulative reformulations."""
    desc = B.desc_like(x, p.k, p.levels)
    y = torch.empty_like(x) if y is None else y
    nb = B.wtconv_variant_workspace_size(desc, variant)
    buf, size = (ws or Workspace(x.device)).get(nb)
    B.wtconv_forward_variant(desc, variant, x, p.w0, p.b0, p.s0, p.wl if p.levels else None,
                             p.sl if p.levels else None, y, buf, size, stream)
    return y


def backward_data(dy: torch.Tensor, p: Params, f: Folded | None = None,
                  ws: Workspace | None = None, dx: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    desc = B.desc_like(dy, p.k, p.levels)
    f = f or fold(p, desc, stream)
    dx = torch.empty_like(dy) if dx is None else dx
    _, nb, _ = B.wtconv_workspace_size(desc)
    buf, size = (ws or Workspace(dy.device)).get(nb)
    B.wtconv_backward_data(desc, dy, f.w0f, f.wlf if p.levels else None, dx, buf, size, stream)
    return dx


def _grad_buffers(p: Params) -> dict:
    return {
        "dw0": torch.empty_like(p.w0),
        "db0": torch.empty_like(p.s0),
        "ds0": torch.empty_like(p.s0),
        "dwl": torch.empty_like(p.wl),
        "dsl": torch.empty_like(p.sl),
    }


def backward_weight(x: torch.Tensor, dy: torch.Tensor, p: Params, ws: Workspace | None = None,
                    out: dict | None = None, stream=None) -> dict:
    desc = B.desc_like(x, p.k, p.levels)
    g = out or _grad_buffers(p)
    _, _, nb = B.wtconv_workspace_size(desc)
    buf, size = (ws or Workspace(x.device)).get(nb)
    lv = p.levels > 0
    B.wtconv_backward_weight(desc, x, dy, p.w0, p.b0, p.s0, p.wl if lv else None,
                             p.sl if lv else None, g["dw0"], g["db0"], g["ds0"],
                             g["dwl"] if lv else None, g["dsl"] if lv else None, buf, size,
                             stream)
    return g


def backward(x: torch.Tensor, dy: torch.Tensor, p: Params, f: Folded | None = None,
             ws: Workspace | None = None, out: dict | None = None, stream=None) -> dict:
    """dx and all parameter gradients in one call (wtconv_backward)."""
    desc = B.desc_like(x, p.k, p.levels)
    f = f or fold(p, desc, stream)
    g = out or _grad_buffers(p)
    if "dx" not in g:
        g["dx"] = torch.empty_like(dy)
    _, nbd, nbw = B.wtconv_workspace_size(desc)
    buf, size = (ws or Workspace(x.device)).get(max(nbd, nbw))
    lv = p.levels > 0
    B.wtconv_backward(desc, x, dy, f.w0f, f.wlf if lv else None, p.w0, p.b0, p.s0,
                      p.wl if lv else None, p.sl if lv else None, g["dx"], g["dw0"], g["db0"],
                      g["ds0"], g["dwl"] if lv else None, g["dsl"] if lv else None, buf, size,
                      stream)
    return g
