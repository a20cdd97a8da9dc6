"""Element-traffic and arithmetic models of the WTConv layer (host-side reporting only).

From "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation":
  * Eq. 2  -- traffic of the reference (framework-primitive) implementation,
              Q_ref = 7N + (43/3) N (1 - 4^-L) elements per forward pass;
  * Eq. 10 -- traffic of the paper's fused implementation,
              Q_fused = 4N + (13/3) N (1 - 4^-L) - N 4^-L;
  * Eq. 3  -- multiply-accumulates of the reference, MAC = N [k^2 + (k^2 + 8)(4/3)(1 - 4^-L)].
All are in units of N = B*C*H*W. Table 1 of the paper prints Eq. 2 / Eq. 10 for L = 1..5.

The algorithmic work used for this library's roofline (see ``algorithmic``) is defined
here once: the ideal single-read/single-write bytes of each pass and the FLOPs of its
depthwise convolutions (2 per multiply-accumulate; Haar butterflies and the synthesis
sum are not counted).
"""
from __future__ import annotations


def level_fraction(levels: int) -> float:
    """sum_{l=1..L} N_l / N with N_l = N / 4^(l-1): (4/3)(1 - 4^-L)."""
    return 4.0 / 3.0 * (1.0 - 4.0 ** (-levels))


def q_ref(levels: int) -> float:
    """Eq. 2: reference-implementation elements per forward pass, per input element."""
    return 7.0 + 43.0 / 3.0 * (1.0 - 4.0 ** (-levels))


def q_fused(levels: int) -> float:
    """Eq. 10: the paper's fused-implementation elements per forward pass, per element."""
    return 4.0 + 13.0 / 3.0 * (1.0 - 4.0 ** (-levels)) - 4.0 ** (-levels)


def q_variant(variant: int, levels: int) -> float:
    """Elements per input element that each staged pipeline of include/wtconv_ablation.h
    moves through HBM in one forward pass, counted stage by stage as in §3.1 and §4.4
    (each stage reads its inputs once and writes its outputs once; weights negligible).

    S = sum_l N_l / N, d = N_L / (4N) = 4^-L (the deepest level's low-pass band):
      0 reference            7 + (6 + 19/4) S - d   (Eq. 2, except that the deepest level's
                             low-pass add has no coarser level to add: it reads one operand)
      1 fused analysis       7 + (9/4 + 19/4) S - 2d (per level: read the carrier, write Z and,
                             except at the deepest level, the raw low-pass carrier)
      2 collapsed synthesis  8 + (9/4 + 1) S - d    (one synthesis pass reads every Z^(l) and
                             writes the level sum; base conv, scale and add stay separate)
      3 folded               4 + 13/4 S - d         (Eq. 10: the pages' fused plan)
    """
    if levels == 0:  # base conv, scale, and the final add with nothing to add (2N each)
        return 2.0 if variant == 3 else 6.0
    S = level_fraction(levels)
    d = 4.0 ** (-levels)
    if variant == 0:
        return 7.0 + (6.0 + 19.0 / 4.0) * S - d
    if variant == 1:
        return 7.0 + 7.0 * S - 2.0 * d
    if variant == 2:
        return 8.0 + 13.0 / 4.0 * S - d
    if variant == 3:
        return 4.0 + 13.0 / 4.0 * S - d
    raise ValueError(variant)


def mac_ref(k: int, levels: int) -> float:
    """Eq. 3: multiply-accumulates per input element of the reference implementation."""
    return k * k + (k * k + 8) * level_fraction(levels)


def conv_macs(k: int, levels: int) -> float:
    """Depthwise-convolution multiply-accumulates per input element of one pass:
    the base k x k plus k x k on all four subbands at every level."""
    return k * k * (1.0 + level_fraction(levels))


def algorithmic(k: int, levels: int, elem_bytes: int) -> dict:
    """Per-input-element algorithmic work of each pass (the roofline's numerators).

    forward:          read X, write Y                    -> 2 e bytes
    backward_data:    read dY, write dX                  -> 2 e bytes
    backward_weight:  read X and dY (parameter grads are O(C k^2), negligible) -> 2 e
    Each pass does conv_macs(k, L) multiply-accumulates = 2 * conv_macs FLOPs.
    """
    flops = 2.0 * conv_macs(k, levels)
    return {
        "forward": {"bytes": 2.0 * elem_bytes, "flops": flops},
        "backward_data": {"bytes": 2.0 * elem_bytes, "flops": flops},
        "backward_weight": {"bytes": 2.0 * elem_bytes, "flops": flops},
    }
