"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test names the passage of "Fast and Memory-Efficient Wavelet Convolutions via
I/O-Aware Reformulation" (Aflalo et al.) that fixes the expected value. Together they are
chosen so that a plausible slip in the oracle -- a dropped term, a wrong sign or index, a
transposed operand, a missing scale -- fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from depthwise_receptive_field_gb300 import iomodel
from depthwise_receptive_field_gb300.inputs import make_inputs, shape_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    return np.loadtxt(os.path.join(GOLDEN, name), comments="#", ndmin=2)


def _params(n, c, h, w, k, L, seed, bias_and_scale=True):
    return make_inputs(shape_workload(n, c, h, w, k, L, "f32", seed), bias_and_scale=bias_and_scale)


# ---------------------------------------------------------------------------------------
# Haar building blocks: Prop. 1, Eq. 5, Eq. 12/13
# ---------------------------------------------------------------------------------------

def test_haar_worked_2x2_block(oracle_lib):
    """Eq. 5 on [a b; c d] = [1 2; 3 4]: LL = 5, LH = -2, HL = -1, HH = 0 (by hand)."""
    out = oracle.haar_analysis(np.array([[1.0, 2.0], [3.0, 4.0]]))
    assert out[:, 0, 0].tolist() == [5.0, -2.0, -1.0, 0.0]


def test_haar_matrix_matches_prop1(oracle_lib):
    """The oracle's analysis, applied to the four unit 2x2 blocks, is the matrix of
    Prop. 1; that matrix is symmetric and squares to the identity."""
    cols = []
    for e in range(4):
        blk = np.zeros(4)
        blk[e] = 1.0
        cols.append(oracle.haar_analysis(blk.reshape(2, 2))[:, 0, 0])
    Hm = np.stack(cols, axis=1)  # rows = bands, columns = (a, b, c, d)
    expected = _golden("haar_matrix_prop1.txt") / 2.0
    assert np.array_equal(Hm, expected)
    assert np.array_equal(Hm, Hm.T)
    assert np.array_equal(Hm @ Hm, np.eye(4))


def test_synthesis_sign_table_eq13(oracle_lib):
    """A unit coefficient in one band, synthesized, shows the sign pattern of Eq. 13
    with the 1/2 of Eq. 12; LL is + everywhere."""
    table = _golden("synthesis_signs_eq13.txt")
    for band in range(4):
        coeff = np.zeros((4, 1, 1))
        coeff[band, 0, 0] = 1.0
        img = oracle.haar_synthesis(coeff)
        for ry, rx, s_lh, s_hl, s_hh in table:
            expect = 0.5 * [1.0, s_lh, s_hl, s_hh][band]
            assert img[int(ry), int(rx)] == expect


def test_synthesis_inverts_analysis(oracle_lib):
    """Prop. 1 (H^-1 = H^T = H): synthesis(analysis(x)) == x, exactly for integers."""
    rng = np.random.default_rng(0)
    img = rng.integers(-50, 50, size=(6, 10)).astype(np.float64)
    assert np.array_equal(oracle.haar_synthesis(oracle.haar_analysis(img)), img)
    coeff = rng.integers(-50, 50, size=(4, 3, 5)).astype(np.float64)
    assert np.array_equal(oracle.haar_analysis(oracle.haar_synthesis(coeff)), coeff)


def test_dwconv_matches_library(oracle_lib):
    """Depthwise convolution = zero-padded 'same' cross-correlation, as torch's conv2d."""
    rng = np.random.default_rng(1)
    for k, (h, w) in [(1, (4, 5)), (3, (7, 6)), (5, (9, 11)), (7, (5, 4))]:
        img = rng.standard_normal((h, w))
        wt = rng.standard_normal((k, k))
        ref = F.conv2d(torch.from_numpy(img)[None, None], torch.from_numpy(wt)[None, None],
                       padding=(k - 1) // 2)[0, 0].numpy()
        np.testing.assert_allclose(oracle.dwconv(img, wt), ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# Algorithm 1 against library primitives (the reference implementation's own style, §3.1)
# ---------------------------------------------------------------------------------------

_HAAR_FILTERS = 0.5 * torch.tensor(
    [[[1, 1], [1, 1]], [[1, 1], [-1, -1]], [[1, -1], [1, -1]], [[1, -1], [-1, 1]]],
    dtype=torch.float64)  # Eq. 5 as 2x2 stride-2 filters, bands (LL, LH, HL, HH)


def _alg1_torch(x, w0, b0, s0, wl, sl, L):
    """Algorithm 1 written with framework primitives, as §3.1 describes the reference:
    Haar analysis as a grouped stride-2 conv2d with +-1/2 filters, the level filter as a
    depthwise conv over the 4C-channel tensor, a scale multiply, LL slicing, and the
    synthesis as the grouped conv_transpose2d. A carrier with an odd side is padded with
    one zero row / column (F.pad) before its analysis and each synthesis output is cropped
    back to the carrier's size. Float64, differentiable by autograd."""
    N, C, H, W = x.shape
    k = w0.shape[-1]
    r = (k - 1) // 2
    haar = _HAAR_FILTERS.unsqueeze(1).repeat(C, 1, 1, 1)  # [4C, 1, 2, 2]
    cur = x
    Z = []
    sizes = []
    for l in range(L):
        sizes.append(cur.shape[-2:])
        cur = F.pad(cur, (0, cur.shape[-1] % 2, 0, cur.shape[-2] % 2))
        Y = F.conv2d(cur, haar, stride=2, groups=C)  # channel 4c + b
        Cv = F.conv2d(Y, wl[l].reshape(4 * C, 1, k, k), padding=r, groups=4 * C)
        Z.append(Cv * sl[l].reshape(1, 4 * C, 1, 1))
        cur = Y[:, 0::4]
    R = None
    for l in reversed(range(L)):
        Zl = Z[l]
        if R is not None:
            add = torch.zeros_like(Zl)
            add[:, 0::4] = R
            Zl = Zl + add
        R = F.conv_transpose2d(Zl, haar, stride=2, groups=C)
        R = R[:, :, :sizes[l][0], :sizes[l][1]]
    base = F.conv2d(x, w0.reshape(C, 1, k, k), padding=r, groups=C) + b0.reshape(1, C, 1, 1)
    out = s0.reshape(1, C, 1, 1) * base
    return out + R if R is not None else out


CASES = [  # n, c, h, w, k, L
    (2, 3, 16, 8, 5, 1),
    (1, 2, 16, 16, 3, 2),
    (2, 2, 32, 16, 5, 3),
    (1, 3, 8, 24, 1, 2),
    (1, 2, 16, 16, 7, 4),
    (2, 3, 12, 10, 5, 0),
    (1, 2, 13, 11, 5, 2),   # odd sides: carriers padded at every level
    (2, 2, 7, 9, 3, 3),     # 7 -> 4 -> 2 -> 1 rows, 9 -> 5 -> 3 -> 2 columns
    (1, 1, 6, 5, 1, 2),     # 6 -> 3 -> 2: an odd carrier at level 2 only
]


@pytest.mark.parametrize("n,c,h,w,k,L", CASES)
@pytest.mark.parametrize("mode", ["cascade", "closed"])
def test_forward_matches_library_primitives(oracle_lib, n, c, h, w, k, L, mode):
    p = _params(n, c, h, w, k, L, seed=10 + L)
    t = {key: (v.double() if v is not None else None) for key, v in p.items()}
    ref = _alg1_torch(t["x"], t["w0"], t["b0"], t["s0"], t["wl"], t["sl"], L).numpy()
    y = oracle.forward(p["x"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L, mode=mode)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("n,c,h,w,k,L", CASES)
def test_backward_matches_library_autograd(oracle_lib, n, c, h, w, k, L):
    p = _params(n, c, h, w, k, L, seed=20 + L)
    t = {key: v.double().clone().requires_grad_(True) for key, v in p.items() if v is not None}
    dy = p["dy"].double()
    out = _alg1_torch(t["x"], t["w0"], t["b0"], t["s0"], t["wl"], t["sl"], L)
    out.backward(dy)
    g = oracle.backward(p["x"], p["dy"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    pairs = [("dx", "x"), ("dw0", "w0"), ("db0", "b0"), ("ds0", "s0")]
    if L > 0:
        pairs += [("dwl", "wl"), ("dsl", "sl")]
    for mine, theirs in pairs:
        ref = t[theirs].grad.numpy()
        np.testing.assert_allclose(g[mine], ref, rtol=0,
                                   atol=1e-11 * max(1.0, np.abs(ref).max()), err_msg=mine)


# ---------------------------------------------------------------------------------------
# Closed forms, special cases and invariants
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("h,w,L", [(13, 11, 2), (7, 9, 3), (5, 6, 2), (17, 3, 2)])
def test_odd_sizes_equal_padding_the_input(oracle_lib, h, w, L):
    """Zero-padding every odd carrier is the same operator as zero-padding X once to a
    multiple of 2^L and cropping the output: the padded region of each carrier is exactly
    the analysis of zeros, and the level coefficients that reach the cropped output sit at
    (y >> l, x >> l) inside the padded grid. Gradients: dX is the cropped dX of the padded
    problem with dY zero-padded; parameter gradients are equal."""
    n, c, k = 2, 2, 5
    p = _params(n, c, h, w, k, L, seed=40 + h + w)
    m = 1 << L
    hp, wp = -(-h // m) * m, -(-w // m) * m
    xp = np.zeros((n, c, hp, wp)); xp[:, :, :h, :w] = p["x"]
    gp = np.zeros((n, c, hp, wp)); gp[:, :, :h, :w] = p["dy"]
    for mode in ("cascade", "closed"):
        y = oracle.forward(p["x"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L, mode=mode)
        yp = oracle.forward(xp, p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L, mode=mode)
        np.testing.assert_allclose(y, yp[:, :, :h, :w], rtol=0, atol=1e-12)
    g = oracle.backward(p["x"], p["dy"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    gpad = oracle.backward(xp, gp, p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    np.testing.assert_allclose(g["dx"], gpad["dx"][:, :, :h, :w], rtol=0, atol=1e-11)
    for key in ("dw0", "db0", "ds0", "dwl", "dsl"):
        np.testing.assert_allclose(g[key], gpad[key], rtol=0,
                                   atol=1e-11 * max(1.0, np.abs(gpad[key]).max()), err_msg=key)


def _delta(k):
    d = np.zeros((k, k))
    d[(k - 1) // 2, (k - 1) // 2] = 1.0
    return d


@pytest.mark.parametrize("L", [1, 2, 3, 4])
def test_exact_reconstruction(oracle_lib, L):
    """W^(0) = 0; identity kernels with unit scale on every band of level L and on the
    high bands of levels < L, zero on their LL bands: the cascade telescopes to Y = X
    exactly (integers, fp64). The carried R^(l+1) replaces the zeroed LL (Alg. 1 line 10)."""
    n, c, h, w, k = 2, 3, 32, 48, 5
    rng = np.random.default_rng(L)
    x = rng.integers(-100, 100, size=(n, c, h, w)).astype(np.float64)
    w0 = np.zeros((c, k, k))
    s0 = np.ones(c)
    wl = np.zeros((L, c, 4, k, k))
    for l in range(L):
        for b in range(4):
            if b == 0 and l < L - 1:
                continue
            wl[l, :, b] = _delta(k)
    sl = np.ones((L, c, 4))
    for mode in ("cascade", "closed"):
        y = oracle.forward(x, w0, None, s0, wl, sl, L, mode=mode)
        assert np.array_equal(y, x), mode


def test_identity_on_every_band_is_not_identity(oracle_lib):
    """With identity on LL too and L = 2, the level-2 reconstruction is added on top of
    the raw LL band, so Y = X + (an extra copy of the level-1 LL content) != X."""
    n, c, h, w, k, L = 1, 1, 8, 8, 3, 2
    x = np.arange(64, dtype=np.float64).reshape(1, 1, 8, 8)
    wl = np.zeros((L, c, 4, k, k))
    wl[:, :, :] = _delta(k)
    y = oracle.forward(x, np.zeros((c, k, k)), None, np.ones(c), wl, np.ones((L, c, 4)), L)
    assert not np.array_equal(y, x)


def test_level0_is_plain_depthwise_conv(oracle_lib):
    """L = 0: Y = s0 * (X *dw W0 + b) = torch's grouped conv2d (a textbook routine)."""
    p = _params(2, 4, 9, 13, 5, 0, seed=3)
    x = p["x"].double()
    ref = F.conv2d(x, p["w0"].double().unsqueeze(1), bias=p["b0"].double(), padding=2, groups=4)
    ref = ref * p["s0"].double().reshape(1, 4, 1, 1)
    y = oracle.forward(p["x"], p["w0"], p["b0"], p["s0"], None, None, 0)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_closed_form_equals_cascade_bit_exact(oracle_lib, L):
    """Prop. 2 / App. A: Eq. 7 equals the cascade of Alg. 1 lines 8-11. With small
    integers and power-of-two parameters every intermediate is exact in fp64, so the two
    evaluation orders must agree bit for bit."""
    rng = np.random.default_rng(100 + L)
    n, c, k = 2, 3, 5
    h = w = 2 ** L * 3
    x = rng.integers(-16, 16, size=(n, c, h, w)).astype(np.float64)
    pick = np.array([0.0, 1.0, -1.0, 0.5, -0.5, 0.25, -0.25, 2.0])
    w0 = rng.choice(pick, size=(c, k, k))
    wl = rng.choice(pick, size=(L, c, 4, k, k))
    sl = rng.choice(np.array([0.5, 1.0, 2.0, 0.25]), size=(L, c, 4))
    s0 = rng.choice(np.array([0.5, 1.0, 2.0]), size=c)
    b0 = rng.choice(pick, size=c)
    a = oracle.forward(x, w0, b0, s0, wl, sl, L, mode="cascade")
    b = oracle.forward(x, w0, b0, s0, wl, sl, L, mode="closed")
    assert np.array_equal(a, b)


def test_scale_folding_forward(oracle_lib):
    """§4.3 Eq. 8: the forward with (W, s, b) equals the forward with W~ = s W, s = 1,
    b~ = s0 b and unit base scale."""
    L = 3
    p = _params(2, 3, 16, 16, 5, L, seed=7)
    y = oracle.forward(p["x"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    w0f = p["s0"].double()[:, None, None] * p["w0"].double()
    b0f = p["s0"].double() * p["b0"].double()
    wlf = p["sl"].double()[..., None, None] * p["wl"].double()
    yf = oracle.forward(p["x"], w0f, b0f, torch.ones(3), wlf, torch.ones(L, 3, 4), L)
    np.testing.assert_allclose(y, yf, rtol=0, atol=1e-12 * np.abs(y).max())


def test_eq9_gradient_unfolding(oracle_lib):
    """§4.3 Eq. 9: gradients of the unfolded parameters equal s * dW~, s * db~ and
    <dW~, W> + db~ b computed from the gradients of the folded parameters."""
    L = 2
    p = _params(2, 3, 16, 16, 5, L, seed=8)
    lit = oracle.backward(p["x"], p["dy"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    s0, b0, w0 = p["s0"].double().numpy(), p["b0"].double().numpy(), p["w0"].double().numpy()
    sl, wl = p["sl"].double().numpy(), p["wl"].double().numpy()
    w0f = s0[:, None, None] * w0
    wlf = sl[..., None, None] * wl
    fol = oracle.backward(p["x"], p["dy"], w0f, s0 * b0, np.ones(3), wlf, np.ones((L, 3, 4)), L)
    tol = dict(rtol=0, atol=1e-10)
    np.testing.assert_allclose(lit["dw0"], s0[:, None, None] * fol["dw0"], **tol)
    np.testing.assert_allclose(lit["db0"], s0 * fol["db0"], **tol)
    np.testing.assert_allclose(
        lit["ds0"], (fol["dw0"] * w0).sum(axis=(1, 2)) + fol["db0"] * b0, **tol)
    np.testing.assert_allclose(lit["dwl"], sl[..., None, None] * fol["dwl"], **tol)
    np.testing.assert_allclose(lit["dsl"], (fol["dwl"] * wl).sum(axis=(3, 4)), **tol)
    np.testing.assert_allclose(lit["dx"], fol["dx"], **tol)


@pytest.mark.parametrize("L", [0, 1, 2, 3])
def test_backward_data_is_rotated_forward(oracle_lib, L):
    """Reading of the backward-data step: by Eq. 1 (the adjoint of analysis is synthesis
    and vice versa) and the adjoint of cross-correlation being correlation with the
    180-degree-rotated kernel, dX equals the forward applied to dY with every folded
    kernel rotated, unit scales and no bias."""
    p = _params(2, 3, 16, 16, 5, L, seed=30 + L)
    lit = oracle.backward(p["x"], p["dy"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    s0 = p["s0"].double()
    w0r = torch.flip(s0[:, None, None] * p["w0"].double(), dims=(-2, -1))
    wlr = torch.flip(p["sl"].double()[..., None, None] * p["wl"].double(), dims=(-2, -1))
    dx = oracle.forward(p["dy"], w0r, None, torch.ones(3), wlr, torch.ones(L, 3, 4), L)
    np.testing.assert_allclose(lit["dx"], dx, rtol=0, atol=1e-11 * np.abs(dx).max())


@pytest.mark.parametrize("L", [1, 2, 3])
def test_finite_differences(oracle_lib, L):
    """Central differences of <dY, F(params)> in fp64 on a tiny layer. F is linear in X,
    W^(0), b, W^(l) and in s^(0), s^(l) separately, so central differences are exact up
    to rounding."""
    n, c, h, w, k = 1, 2, 8, 8, 3
    p = _params(n, c, h, w, k, L, seed=40 + L)
    base = {key: p[key].double().numpy().copy() for key in ("x", "w0", "b0", "s0", "wl", "sl")}
    dy = p["dy"].double().numpy()
    g = oracle.backward(base["x"], dy, base["w0"], base["b0"], base["s0"], base["wl"],
                        base["sl"], L)
    names = {"x": "dx", "w0": "dw0", "b0": "db0", "s0": "ds0", "wl": "dwl", "sl": "dsl"}
    eps = 1e-6

    def loss(q):
        y = oracle.forward(q["x"], q["w0"], q["b0"], q["s0"], q["wl"], q["sl"], L)
        return float((y * dy).sum())

    rng = np.random.default_rng(L)
    for key, gname in names.items():
        arr = base[key]
        flat_idx = range(arr.size) if arr.size <= 80 else rng.choice(arr.size, 80, replace=False)
        for fi in flat_idx:
            idx = np.unravel_index(fi, arr.shape)
            q = {kk: vv.copy() for kk, vv in base.items()}
            q[key][idx] += eps
            lp = loss(q)
            q[key][idx] -= 2 * eps
            lm = loss(q)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (key, idx, fd, g[gname][idx])


@pytest.mark.parametrize("shape", [(2, 3, 20, 28, 5, 3), (1, 2, 32, 32, 7, 4),
                                   (1, 2, 24, 40, 1, 2)])
def test_gradients_along_whole_tensor_directions(oracle_lib, shape):
    """Algorithm 1 is affine in each of X, W^(0), b, s^(0), W^(l), s^(l) with the others
    held (every stage is a convolution, a Haar step, a scale or a sum), so for a random
    direction D of one of them <dY, F(P + D) - F(P)> equals <dP, D> up to rounding, at
    sizes and odd carrier sides that finite differences element by element do not reach."""
    n, c, h, w, k, L = shape
    p = _params(n, c, h, w, k, L, seed=90 + k)
    base = {key: p[key].double().numpy().copy() for key in ("x", "w0", "b0", "s0", "wl", "sl")}
    dy = p["dy"].double().numpy()
    g = oracle.backward(base["x"], dy, base["w0"], base["b0"], base["s0"], base["wl"],
                        base["sl"], L)
    names = {"x": "dx", "w0": "dw0", "b0": "db0", "s0": "ds0", "wl": "dwl", "sl": "dsl"}
    y0 = oracle.forward(base["x"], base["w0"], base["b0"], base["s0"], base["wl"], base["sl"], L)
    rng = np.random.default_rng(k)
    for key, gname in names.items():
        d = rng.standard_normal(base[key].shape)
        q = dict(base)
        q[key] = base[key] + d
        y1 = oracle.forward(q["x"], q["w0"], q["b0"], q["s0"], q["wl"], q["sl"], L)
        lhs = float(((y1 - y0) * dy).sum())
        rhs = float((g[gname] * d).sum())
        scale = float((np.abs(y1 - y0) * np.abs(dy)).sum())
        assert abs(lhs - rhs) <= 1e-12 * scale, (key, lhs, rhs)


def _operator_matrix(fn, size):
    cols = []
    for e in range(size):
        v = np.zeros(size)
        v[e] = 1.0
        cols.append(fn(v).ravel())
    return np.stack(cols, axis=1)


def test_bruteforce_operator_transpose(oracle_lib):
    """Brute force on an 8x8 plane: build the dense forward operator T column by column
    from unit inputs (b = 0); the backward-data operator built the same way from unit
    output gradients must be exactly T^T (up to rounding). Also checks the adjoint dot
    identity <F(X), dY> = <X, dX(dY)> on random vectors."""
    L, k = 3, 3
    p = _params(1, 1, 8, 8, k, L, seed=50)
    prm = dict(w0=p["w0"], b0=None, s0=p["s0"], wl=p["wl"], sl=p["sl"])

    def fwd(v):
        return oracle.forward(v.reshape(1, 1, 8, 8), levels=L, **prm)

    def bwd(v):
        return oracle.backward(np.zeros((1, 1, 8, 8)), v.reshape(1, 1, 8, 8), levels=L,
                               **prm)["dx"]

    T = _operator_matrix(fwd, 64)
    B = _operator_matrix(bwd, 64)
    np.testing.assert_allclose(B, T.T, rtol=0, atol=1e-13)
    rng = np.random.default_rng(5)
    xv, gv = rng.standard_normal(64), rng.standard_normal(64)
    assert abs(float(fwd(xv).ravel() @ gv) - float(xv @ bwd(gv).ravel())) < 1e-12


def test_receptive_field_support(oracle_lib):
    """§1 / Eq. 7: output (y, x) depends only on the base k x k window and, at level l, on
    the input rows and columns of the coarse window around (y >> l, x >> l):
    [2^l((y>>l) - R), 2^l((y>>l) + R + 1) - 1]. The bounding box of the dependence is
    exactly the largest of these windows (clipped to the plane)."""
    L, k, S = 3, 3, 32
    r = (k - 1) // 2
    p = _params(1, 1, S, S, k, L, seed=51)
    prm = dict(w0=p["w0"], b0=None, s0=p["s0"], wl=p["wl"], sl=p["sl"])
    rng = np.random.default_rng(9)
    T = _operator_matrix(lambda v: oracle.forward(v.reshape(1, 1, S, S), levels=L, **prm), S * S)
    for out_idx in rng.choice(S * S, 40, replace=False):
        y, x = divmod(int(out_idx), S)
        allowed = np.zeros((S, S), dtype=bool)
        allowed[max(0, y - r):y + r + 1, max(0, x - r):x + r + 1] = True
        lo_y = lo_x = S
        hi_y = hi_x = -1
        for l in range(1, L + 1):
            ys = (2 ** l) * ((y >> l) - r), (2 ** l) * ((y >> l) + r + 1) - 1
            xs = (2 ** l) * ((x >> l) - r), (2 ** l) * ((x >> l) + r + 1) - 1
            allowed[max(0, ys[0]):ys[1] + 1, max(0, xs[0]):xs[1] + 1] = True
            lo_y, hi_y = min(lo_y, max(0, ys[0])), max(hi_y, min(S - 1, ys[1]))
            lo_x, hi_x = min(lo_x, max(0, xs[0])), max(hi_x, min(S - 1, xs[1]))
        dep = np.abs(T[out_idx].reshape(S, S)) > 1e-14
        assert not (dep & ~allowed).any()
        rows, cols = np.nonzero(dep)
        assert (rows.min(), rows.max(), cols.min(), cols.max()) == (lo_y, hi_y, lo_x, hi_x)


def test_batch_and_channel_independence(oracle_lib):
    """Depthwise structure: the forward of one (n, c) plane depends only on that plane and
    channel c's parameters (what the sampled full-size parity checks rely on)."""
    L = 2
    p = _params(3, 4, 16, 16, 5, L, seed=60)
    y = oracle.forward(p["x"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], L)
    sub = oracle.forward(p["x"][1:2, 2:3], p["w0"][2:3], p["b0"][2:3], p["s0"][2:3],
                         p["wl"][:, 2:3], p["sl"][:, 2:3], L)
    assert np.array_equal(y[1:2, 2:3], sub)


def test_invalid_arguments_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle.forward(np.zeros((1, 1, 6, 6)), np.zeros((1, 4, 4)), None, np.ones(1),
                       np.zeros((1, 1, 4, 4, 4)), np.ones((1, 1, 4)), 1)  # even k
    with pytest.raises(ValueError):
        oracle.forward(np.zeros((1, 1, 6, 6)), np.zeros((1, 3, 3)), None, np.ones(1),
                       np.zeros((31, 1, 4, 3, 3)), np.ones((31, 1, 4)), 31)  # L > 30


# ---------------------------------------------------------------------------------------
# The I/O and arithmetic models (host-side reporting)
# ---------------------------------------------------------------------------------------

def test_traffic_model_reproduces_table1():
    for L, qr, qf, ratio in _golden("traffic_table1.txt"):
        L = int(L)
        assert round(iomodel.q_ref(L), 2) == pytest.approx(qr, abs=0.011)
        assert round(iomodel.q_fused(L), 2) == pytest.approx(qf, abs=0.011)
        assert round(iomodel.q_ref(L) / iomodel.q_fused(L), 2) == pytest.approx(ratio, abs=0.011)
    assert iomodel.q_ref(60) / iomodel.q_fused(60) == pytest.approx(64 / 25)  # Eq. 11 limit


def test_mac_model_reproduces_section1():
    for k, L, macs in _golden("mac_counts_sec1.txt"):
        assert iomodel.mac_ref(int(k), int(L)) == pytest.approx(macs, abs=0.05)


def test_variant_traffic_models_against_the_pages():
    """The staged pipelines' traffic counts reduce to the pages' own formulas: the folded
    variant is Eq. 10 exactly, the reference is Eq. 2 less the one operand the deepest
    level's low-pass add does not read, and every reformulation lowers the count."""
    for L in range(1, 8):
        assert iomodel.q_variant(3, L) == pytest.approx(iomodel.q_fused(L), abs=1e-12)
        assert iomodel.q_variant(0, L) == pytest.approx(iomodel.q_ref(L) - 4.0 ** (-L),
                                                        abs=1e-12)
        qs = [iomodel.q_variant(v, L) for v in range(4)]
        assert qs == sorted(qs, reverse=True) and len(set(qs)) == 4
    # Table 1 values at L = 1 (17.75N reference, 7.00N fused)
    assert iomodel.q_variant(3, 1) == pytest.approx(7.0)
    assert iomodel.q_variant(0, 1) + 0.25 == pytest.approx(17.75)
