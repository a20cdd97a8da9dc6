"""The C-ABI library builds, loads without a GPU, exports every declared symbol, and its
host-side validation and workspace sizing behave as include/wtconv.h documents. No CUDA
kernel is launched here: every call below returns before reaching the device."""
import ctypes

import pytest

from depthwise_receptive_field_gb300 import binding as B
from depthwise_receptive_field_gb300.inputs import WORKLOADS


@pytest.fixture(scope="module")
def lib():
    return B.load_library()


def test_exports_every_declared_symbol(lib):
    names = B.declared_functions()
    assert len(names) >= 8, names
    for name in names:
        assert hasattr(lib, name), name


def test_header_declares_the_method_entry_points():
    names = set(B.declared_functions())
    for required in ("wtconv_forward", "wtconv_backward_data", "wtconv_backward_weight",
                     "wtconv_fold_scales", "wtconv_workspace_size", "wtconv_status_string"):
        assert required in names


def test_status_strings(lib):
    for s in range(6):
        assert B.status_string(s).startswith("WT_")
    assert "unknown" in B.status_string(99)


BAD = [
    dict(k=4),              # even kernel
    dict(k=0),
    dict(levels=-1),
    dict(levels=13),
    dict(h=0),
    dict(w=-3),
    dict(n=0),
    dict(c=0),
    dict(io=7),
]


@pytest.mark.parametrize("override", BAD)
def test_invalid_descriptors_rejected(lib, override):
    base = dict(n=2, c=3, h=32, w=32, k=5, levels=2, io=B.WT_F32)
    base.update(override)
    d = B.wt_desc(**base)
    a = ctypes.c_size_t()
    st = lib.wtconv_workspace_size(ctypes.byref(d), ctypes.byref(a), None, None)
    assert st == B.WT_ERR_INVALID_ARG
    # the compute entry points validate the same way before touching the device
    st = lib.wtconv_forward(ctypes.byref(d), 16, 16, None, 16, 16, None, 0, None)
    assert st == B.WT_ERR_INVALID_ARG


@pytest.mark.parametrize("h,w,L", [(30, 32, 2), (32, 12, 3), (13, 11, 2), (7, 9, 3)])
def test_odd_sides_are_accepted(lib, h, w, L):
    """Sides that are not multiples of 2^L are padded per level (not rejected); the staged
    pipelines, which materialize exact halvings, report them as unsupported."""
    d = B.make_desc(2, 3, h, w, 5, L, B.WT_F32)
    fwd, bwd_d, bwd_w = B.wtconv_workspace_size(d)
    assert fwd == bwd_d and fwd >= 256 and bwd_w > 256
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_variant_workspace_size(d, B.WT_VARIANT_REFERENCE)
    assert e.value.status == B.WT_ERR_UNSUPPORTED


def test_unbuilt_kernel_size_is_unsupported(lib):
    d = B.wt_desc(1, 1, 32, 32, 9, 1, B.WT_F32)
    assert lib.wtconv_workspace_size(ctypes.byref(d), None, None, None) == B.WT_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected(lib):
    d = B.wt_desc(1, 2, 16, 16, 5, 1, B.WT_F32)
    assert lib.wtconv_forward(ctypes.byref(d), None, 16, None, 16, 16, None, 0, None) == 1
    assert lib.wtconv_forward(ctypes.byref(d), 8, 16, None, 16, 16, None, 0, None) == 1
    assert lib.wtconv_backward_data(ctypes.byref(d), 16, 16, 16, 24, None, 0, None) == 1
    assert lib.wtconv_fold_scales(ctypes.byref(d), 16, None, 16, None, 16, 16, None, 16,
                                  None) == 1
    # backward_weight: too small a workspace is reported before any launch
    args = [16] * 13
    st = lib.wtconv_backward_weight(ctypes.byref(d), *args, 0, None)
    assert st in (B.WT_ERR_WORKSPACE, B.WT_ERR_INVALID_ARG)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workspace_sizes_for_workloads(lib, name):
    wl = WORKLOADS[name]
    d = B.make_desc(wl.n, wl.c, wl.h, wl.w, wl.k, wl.levels,
                    B.WT_BF16 if wl.dtype == "bf16" else B.WT_F32)
    fwd, bwd_d, bwd_w = B.wtconv_workspace_size(d)
    # forward / backward-data: a 256-byte status word, the per-channel shared-memory images of
    # the folded weights (base + 2 band pairs per level, each round4(2 k^2) floats), then per
    # resident CTA one scratch slot holding the deep sums and the level-2 subbands, each
    # [H/4][W/4][4] fp32
    assert fwd == bwd_d
    ws_pair = (2 * wl.k * wl.k + 3) // 4 * 4
    img = (wl.c * ws_pair * (1 + 2 * wl.levels) * 4 + 255) // 256 * 256
    if wl.levels < 2:
        assert fwd == 256 + img
    else:
        half = (4 * (wl.h >> 2) * (wl.w >> 2) + 63) // 64 * 64 * 4
        slot = 2 * half
        assert fwd >= 256 + img + slot and (fwd - 256 - img) % slot == 0
        assert fwd <= 256 + img + 2 * 152 * slot  # at most 2 CTAs per SM
    # backward-weight: a 256-byte status word, one partial vector [dW0 | db | dW^(l)] per
    # (channel, image), then per resident CTA (persistent grid, at most 2 per SM) a slot
    # holding the level-2 subbands of X and of dY, each [H/4][W/4][4] fp32 (L >= 2)
    kk = wl.k * wl.k
    per_partial = (kk + 1 + 4 * kk * wl.levels) * 4
    parts = 256 + (wl.c * wl.n * per_partial + 255) // 256 * 256
    if wl.levels < 2:
        assert bwd_w == parts
    else:
        dslot = 2 * ((4 * (wl.h >> 2) * (wl.w >> 2) + 63) // 64 * 64 * 4)
        assert bwd_w >= parts + dslot and (bwd_w - parts) % dslot == 0
        assert bwd_w <= parts + 2 * 152 * dslot


def _header_prototypes():
    """(name, parameter count) of every function the public headers declare."""
    import re
    protos = {}
    for h in B.HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"(?:wt_status|const char\*|int)\s+(wtconv_\w+)\s*\(([^;]*?)\)\s*;",
                             text, flags=re.S):
            args = m.group(2).strip()
            protos[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return protos


def test_binding_arity_matches_header():
    protos = _header_prototypes()
    assert set(protos) == set(B.declared_functions())
    for name, argtypes in B._SIGNATURES.items():
        assert name in protos, name
        assert len(argtypes) == protos[name], (name, len(argtypes), protos[name])


def test_variant_validation(lib):
    d = B.make_desc(2, 3, 64, 64, 5, 2, B.WT_F32)
    sizes = [B.wtconv_variant_workspace_size(d, v) for v in range(4)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    # the reference materializes the most: every stage output of every level
    assert sizes[B.WT_VARIANT_REFERENCE] == max(sizes)
    for bad in (-1, 4):
        with pytest.raises(B.WTConvError) as e:
            B.wtconv_variant_workspace_size(d, bad)
        assert e.value.status == B.WT_ERR_INVALID_ARG
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_variant_workspace_size(B.make_desc(2, 3, 64, 64, 5, 2, B.WT_BF16), 0)
    assert e.value.status == B.WT_ERR_UNSUPPORTED
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_variant_workspace_size(B.make_desc(2, 3, 60, 64, 5, 3, B.WT_F32), 0)
    assert e.value.status == B.WT_ERR_UNSUPPORTED
    # null input pointer: rejected before any launch
    with pytest.raises(B.WTConvError) as e:
        B.wtconv_forward_variant(d, 0, None, 16, None, 16, 16, 16, 16, 256, sizes[0], stream=0)
    assert e.value.status == B.WT_ERR_INVALID_ARG


def test_status_query_and_probe_validate_before_any_device_call(lib):
    """wtconv_workspace_status rejects a NULL workspace, the probe rejects bad sizes and a
    NULL output, and the wait-limit test hook accepts any value; none touches the device."""
    flags = ctypes.c_int(5)
    assert lib.wtconv_workspace_status(None, None, ctypes.byref(flags)) == B.WT_ERR_INVALID_ARG
    assert flags.value == 0
    assert lib.wtconv_fma_probe(0, 10, 1, 256, None) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_fma_probe(4, 0, 1, 256, None) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_fma_probe(4, 10, 1, None, None) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_fma_probe(4, 10, 1, 258, None) == B.WT_ERR_INVALID_ARG  # misaligned
    assert lib.wtconv_testing_set_wait_limit_ns(1000) == B.WT_OK
    assert lib.wtconv_testing_set_wait_limit_ns(0) == B.WT_OK
    assert B.status_string(B.WT_ERR_TIMEOUT).startswith("WT_ERR_TIMEOUT")


def test_phase_clocks_are_absent_from_the_ordinary_library(lib):
    """wtconv_debug_phase_clocks validates its arguments, then reports WT_ERR_UNSUPPORTED:
    the ordinary build has no clock code (only the separate -DWT_PHASE_CLOCKS build does)."""
    buf = (ctypes.c_ulonglong * 32)()
    ptr = ctypes.cast(buf, ctypes.c_void_p)
    assert lib.wtconv_debug_phase_clocks(0, 0, None, 32) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_debug_phase_clocks(0, 0, ptr, 31) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_debug_phase_clocks(2, 0, ptr, 32) == B.WT_ERR_INVALID_ARG
    assert lib.wtconv_debug_phase_clocks(0, 0, ptr, 32) == B.WT_ERR_UNSUPPORTED
    assert lib.wtconv_debug_phase_clocks(1, 1, ptr, 32) == B.WT_ERR_UNSUPPORTED


def test_binding_rejects_tensors_the_abi_cannot_check():
    """The C ABI sees raw pointers only; the binding rejects what a pointer cannot tell:
    a non-contiguous tensor, a wrong dtype or size, a host tensor, a workspace smaller than
    ws_bytes. Raw integer addresses pass through (the ABI's own pointer tests use them)."""
    import torch
    desc = B.make_desc(1, 2, 8, 8, 3, 1, B.WT_F32)
    x = torch.zeros(1, 2, 8, 8)
    for bad, msg in ((x.transpose(2, 3), "contiguous"), (x.double(), "dtype"),
                     (x[:, :1], "elements"), (x, "CUDA")):
        with pytest.raises(ValueError, match=msg):
            B.wtconv_forward(desc, bad, 256, 256, 256, 256)
    with pytest.raises(ValueError, match="dtype"):
        B.wtconv_forward(desc, 256, torch.zeros(2, 3, 3, dtype=torch.float64), 256, 256, 256)
    with pytest.raises(ValueError, match="elements"):
        B.wtconv_backward_weight(desc, 256, 256, torch.zeros(2, 3, 2), 256, 256, 256, 256, 256,
                                 256, 256, 256, 256, None, 0)
    with pytest.raises(ValueError, match="workspace"):
        B.wtconv_forward(desc, 256, 256, 256, 256, 256, torch.zeros(8, dtype=torch.uint8), 64)
