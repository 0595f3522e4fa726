"""Pins for the CPU oracle: checks against closed forms, identities, library
special cases and brute force -- never against the oracle itself.

Each check is chosen so that a plausible slip in the oracle (flipped kernel,
wrong padding side, transposed weight operand, dropped bias, missing tap,
swapped dgrad tap mirror, a wgrad shifted the wrong way) fails at least one of
them; ``test_pins_catch_planted_mistakes`` demonstrates that on mutated copies
of the oracle's own loop nests.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand(*shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def test_centre_delta_reproduces_input():
    C = 5
    x = rand(2, 4, 6, C)
    w = np.zeros((C, 3, 3, C))
    for k in range(C):
        w[k, 1, 1, k] = 1.0
    y = oracle.conv3x3_fwd(x, w)
    assert np.array_equal(y, x)


@pytest.mark.parametrize("r", [0, 1, 2])
@pytest.mark.parametrize("s", [0, 1, 2])
def test_off_centre_delta_shifts_with_zero_fill(r, s):
    # y[h, w] = x[h + r - 1, w + s - 1], zero where that leaves the image
    C = 3
    x = rand(1, 5, 4, C)
    w = np.zeros((C, 3, 3, C))
    for k in range(C):
        w[k, r, s, k] = 1.0
    y = oracle.conv3x3_fwd(x, w)
    xp = np.zeros((1, 7, 6, C))
    xp[:, 1:6, 1:5] = x
    expect = xp[:, r:r + 5, s:s + 4]
    assert np.array_equal(y, expect)


def test_all_ones_kernel_on_constant_input_gives_9_6_4_pattern():
    Cin, cval = 4, 0.75
    H, W = 5, 6
    x = np.full((1, H, W, Cin), cval)
    w = np.ones((2, 3, 3, Cin))
    y = oracle.conv3x3_fwd(x, w)
    nh = np.array([2] + [3] * (H - 2) + [2])
    nw = np.array([2] + [3] * (W - 2) + [2])
    taps = nh[:, None] * nw[None, :]  # 9 interior, 6 edge, 4 corner
    assert taps[0, 0] == 4 and taps[0, 2] == 6 and taps[2, 2] == 9
    for k in range(2):
        assert np.array_equal(y[0, :, :, k], taps * Cin * cval)


def test_one_by_one_special_case_is_a_gemm():
    # only the centre tap is non-zero: y = X W1^T + b, a plain matrix product
    N, H, W, Cin, Cout = 2, 3, 5, 7, 6
    x = rand(N, H, W, Cin)
    w = np.zeros((Cout, 3, 3, Cin))
    w1 = rand(Cout, Cin)
    w[:, 1, 1, :] = w1
    b = rand(Cout)
    y = oracle.conv3x3_fwd(x, w, b)
    expect = (x.reshape(-1, Cin) @ w1.T + b).reshape(N, H, W, Cout)
    assert np.allclose(y, expect, rtol=1e-13, atol=1e-13)


def test_silu_special_values_and_grid():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(-60.0)) < 1e-20
    assert oracle.silu(-1e4) == 0.0
    for z in np.linspace(-12, 12, 97):
        sig = 0.5 * (1.0 + math.tanh(0.5 * z))  # sigmoid via tanh, a different route
        assert oracle.silu(z) == pytest.approx(z * sig, rel=1e-12, abs=1e-15)


def test_silu_epilogue_applies_after_bias():
    x = rand(1, 3, 3, 2)
    w = rand(4, 3, 3, 2)
    b = rand(4)
    z = oracle.conv3x3_fwd(x, w, b, act=0)
    y = oracle.conv3x3_fwd(x, w, b, act=1)
    sig = 0.5 * (1.0 + np.tanh(0.5 * z))
    assert np.allclose(y, z * sig, rtol=1e-12, atol=1e-14)


def test_leaky_relu_special_values_and_epilogue():
    # slope 0.2 below zero, identity at and above zero (the bias + leaky ReLU op)
    assert oracle.lrelu(0.0) == 0.0
    assert oracle.lrelu(3.5) == 3.5
    assert oracle.lrelu(-1.0) == -0.2
    assert oracle.lrelu(-5.0) == -1.0
    for z in np.linspace(-7, 7, 57):
        assert oracle.lrelu(z) == pytest.approx(max(z, 0.2 * z), rel=1e-15, abs=0)
    # applied after the bias: constant input, all-ones kernel, bias chosen so
    # that the interior (9 taps) is positive and the corners (4 taps) negative
    x = np.ones((1, 4, 4, 1))
    w = np.ones((1, 3, 3, 1))
    y = oracle.conv3x3_fwd(x, w, np.array([-5.0]), act=2)
    assert y[0, 1, 1, 0] == 4.0        # 9 - 5
    assert y[0, 0, 1, 0] == 1.0        # 6 - 5
    assert y[0, 0, 0, 0] == -0.2       # 0.2 * (4 - 5)


def test_act_grad_closed_forms_and_finite_differences():
    # SiLU'(0) = 1/2; SiLU' -> 1 above and -> 0 below; leaky ReLU' = 1 or 0.2
    assert oracle.act_grad(1, 0.0) == 0.5
    assert oracle.act_grad(1, 50.0) == pytest.approx(1.0, abs=1e-15)
    assert abs(oracle.act_grad(1, -50.0)) < 1e-18
    assert oracle.act_grad(2, 3.0) == 1.0
    assert oracle.act_grad(2, -3.0) == 0.2
    assert oracle.act_grad(2, 0.0) == 0.2     # the lower one-sided derivative at the kink
    assert oracle.act_grad(0, -7.0) == 1.0
    # central differences of the (separately pinned) activations themselves
    h = 1e-5
    for z in np.linspace(-9, 9, 73):
        fd = (oracle.silu(z + h) - oracle.silu(z - h)) / (2 * h)
        assert oracle.act_grad(1, z) == pytest.approx(fd, rel=1e-8, abs=1e-10)
        if abs(z) > 1e-3:
            fd = (oracle.lrelu(z + h) - oracle.lrelu(z - h)) / (2 * h)
            assert oracle.act_grad(2, z) == pytest.approx(fd, rel=1e-9)
    # SiLU' has one minimum, at the root of its derivative z ~ -2.3994, value ~ -0.0998
    zs = np.linspace(-4, -1, 3001)
    g = np.array([oracle.act_grad(1, z) for z in zs])
    assert zs[np.argmin(g)] == pytest.approx(-2.3994, abs=2e-3)
    assert g.min() == pytest.approx(-0.09984, abs=2e-5)


def _act_elementwise(act, z):
    f = {0: float, 1: oracle.silu, 2: oracle.lrelu}[act]
    return np.vectorize(f)(z)


@pytest.mark.parametrize("act", [1, 2])
def test_dgrad_through_activation_by_finite_differences(act):
    # F(zin) = <v, conv3x3(act(zin), w)>; dF/dzin must equal dgrad_act(v, w, zin)
    N, H, W, Cin, Cout = 1, 3, 4, 2, 3
    zin = rand(N, H, W, Cin)
    w = rand(Cout, 3, 3, Cin)
    v = rand(N, H, W, Cout)
    g = oracle.conv3x3_dgrad_act(v, w, zin, act)

    def F(zz):
        return float(np.sum(v * oracle.conv3x3_fwd(_act_elementwise(act, zz), w)))

    h = 1e-6
    for e in range(zin.size):
        zp = zin.copy().reshape(-1)
        zm = zin.copy().reshape(-1)
        zp[e] += h
        zm[e] -= h
        fd = (F(zp.reshape(zin.shape)) - F(zm.reshape(zin.shape))) / (2 * h)
        assert g.reshape(-1)[e] == pytest.approx(fd, rel=1e-6, abs=1e-8), e


def test_dgrad_through_no_activation_is_plain_dgrad():
    dz = rand(2, 5, 4, 3)
    w = rand(3, 3, 3, 6)
    zin = rand(2, 5, 4, 6)
    assert np.array_equal(oracle.conv3x3_dgrad_act(dz, w, zin, 0), oracle.conv3x3_dgrad(dz, w))


def test_dgrad_through_activation_by_torch_autograd():
    torch = pytest.importorskip("torch")
    N, H, W, Cin, Cout = 2, 5, 6, 4, 3
    zin = rand(N, H, W, Cin)
    w = rand(Cout, 3, 3, Cin)
    dz = rand(N, H, W, Cout)
    for act, fn in ((1, torch.nn.functional.silu),
                    (2, lambda t: torch.nn.functional.leaky_relu(t, negative_slope=0.2))):
        zt = torch.tensor(zin).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
        wt = torch.tensor(w).permute(0, 3, 1, 2).contiguous()
        y = torch.nn.functional.conv2d(fn(zt), wt, stride=1, padding=1)
        y.backward(torch.tensor(dz).permute(0, 3, 1, 2))
        assert np.allclose(oracle.conv3x3_dgrad_act(dz, w, zin, act),
                           zt.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-13)


def test_concatenated_input_splits_into_two_convolutions():
    # conv over concat(xa, xb) = conv(xa, w[..., :Ca]) + conv(xb, w[..., Ca:]) (linearity in x);
    # dgrad's channel c and wgrad's channel c involve only w[..., c] and x[..., c]
    N, H, W, Ca, Cb, Cout = 2, 5, 4, 3, 2, 4
    xa, xb = rand(N, H, W, Ca), rand(N, H, W, Cb)
    w, b, dz = rand(Cout, 3, 3, Ca + Cb), rand(Cout), rand(N, H, W, Cout)
    y = oracle.conv3x3_fwd_cat(xa, xb, w, b)
    ya = oracle.conv3x3_fwd(xa, np.ascontiguousarray(w[..., :Ca]), b)
    yb = oracle.conv3x3_fwd(xb, np.ascontiguousarray(w[..., Ca:]))
    assert np.allclose(y, ya + yb, rtol=1e-12, atol=1e-12)
    dxa, dxb = oracle.conv3x3_dgrad_cat(dz, w, Ca)
    assert np.array_equal(dxa, oracle.conv3x3_dgrad(dz, np.ascontiguousarray(w[..., :Ca])))
    assert np.array_equal(dxb, oracle.conv3x3_dgrad(dz, np.ascontiguousarray(w[..., Ca:])))
    dw, db = oracle.conv3x3_wgrad_cat(xa, xb, dz)
    dwa, dba = oracle.conv3x3_wgrad(xa, dz)
    dwb, _ = oracle.conv3x3_wgrad(xb, dz)
    assert np.array_equal(dw[..., :Ca], dwa) and np.array_equal(dw[..., Ca:], dwb)
    assert np.array_equal(db, dba)
    idx = np.arange(0, y.size, 7)
    assert np.array_equal(oracle.conv3x3_fwd_cat_at(xa, xb, w, b, 0, idx), y.reshape(-1)[idx])
    iw = np.arange(0, dw.size, 5)
    assert np.array_equal(oracle.conv3x3_wgrad_cat_at(xa, xb, dz, iw), dw.reshape(-1)[iw])


# ---------------------------------------------------------------------------
# strided (downsampling) convolution
# ---------------------------------------------------------------------------
def test_strided_with_stride_one_is_the_plain_convolution():
    x, w, b, dz = rand(2, 5, 6, 3), rand(4, 3, 3, 3), rand(4), rand(2, 5, 6, 4)
    assert np.array_equal(oracle.conv3x3_fwd_strided(x, w, b, 1, u=1), oracle.conv3x3_fwd(x, w, b, 1))
    assert np.array_equal(oracle.conv3x3_dgrad_strided(dz, w, 5, 6, u=1), oracle.conv3x3_dgrad(dz, w))
    dw, db = oracle.conv3x3_wgrad_strided(x, dz, u=1)
    rdw, rdb = oracle.conv3x3_wgrad(x, dz)
    assert np.array_equal(dw, rdw) and np.array_equal(db, rdb)


@pytest.mark.parametrize("H,W", [(6, 8), (7, 5), (1, 4), (2, 3)])
def test_stride_two_forward_is_the_plain_output_at_even_positions(H, W):
    x, w, b = rand(2, H, W, 3), rand(4, 3, 3, 3), rand(4)
    y = oracle.conv3x3_fwd_strided(x, w, b, 0, u=2)
    assert y.shape == (2, (H + 1) // 2, (W + 1) // 2, 4)
    assert np.array_equal(y, oracle.conv3x3_fwd(x, w, b)[:, ::2, ::2])


@pytest.mark.parametrize("H,W", [(6, 8), (7, 5), (3, 3)])
def test_stride_two_backward_identities(H, W):
    N, Cin, Cout = 2, 3, 4
    Ho, Wo = (H + 1) // 2, (W + 1) // 2
    x, w, v = rand(N, H, W, Cin), rand(Cout, 3, 3, Cin), rand(N, Ho, Wo, Cout)
    # adjoint: <fwd(x, w), v> = <x, dgrad(v, w)>
    lhs = np.sum(oracle.conv3x3_fwd_strided(x, w, None, 0, u=2) * v)
    rhs = np.sum(x * oracle.conv3x3_dgrad_strided(v, w, H, W, u=2))
    assert lhs == pytest.approx(rhs, rel=1e-12)
    # dgrad = the plain dgrad of v spread onto the even positions of an H x W grid
    up = np.zeros((N, H, W, Cout))
    up[:, ::2, ::2] = v
    assert np.allclose(oracle.conv3x3_dgrad_strided(v, w, H, W, u=2), oracle.conv3x3_dgrad(up, w),
                       rtol=1e-13, atol=1e-13)
    # bilinear: <dw(x, v), V> = <fwd(x, V), v>;  db = sum of v
    dw, db = oracle.conv3x3_wgrad_strided(x, v, u=2)
    V = rand(Cout, 3, 3, Cin)
    assert np.sum(dw * V) == pytest.approx(np.sum(oracle.conv3x3_fwd_strided(x, V, None, 0, u=2) * v),
                                           rel=1e-12)
    assert np.allclose(db, v.sum(axis=(0, 1, 2)), rtol=1e-13, atol=1e-13)
    # sampled variants agree with the full ones
    dx = oracle.conv3x3_dgrad_strided(v, w, H, W, u=2)
    i = np.arange(0, dx.size, 3)
    assert np.array_equal(oracle.conv3x3_dgrad_strided_at(v, w, H, W, 2, i), dx.reshape(-1)[i])
    iw = np.concatenate([np.arange(0, dw.size, 4), dw.size + np.arange(Cout)])
    assert np.array_equal(oracle.conv3x3_wgrad_strided_at(x, v, 2, iw),
                          np.concatenate([dw.reshape(-1), db])[iw])
    y = oracle.conv3x3_fwd_strided(x, w, None, 1, u=2)
    iy = np.arange(0, y.size, 2)
    assert np.array_equal(oracle.conv3x3_fwd_strided_at(x, w, None, 1, 2, iy), y.reshape(-1)[iy])


def test_stride_two_against_torch_float64():
    torch = pytest.importorskip("torch")
    N, H, W, Cin, Cout = 2, 7, 6, 4, 3
    x, w, b = rand(N, H, W, Cin), rand(Cout, 3, 3, Cin), rand(Cout)
    xt = torch.tensor(x).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    wt = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    bt = torch.tensor(b).requires_grad_(True)
    z = torch.nn.functional.conv2d(xt, wt, bt, stride=2, padding=1)
    dz = rand(*z.permute(0, 2, 3, 1).shape)
    z.backward(torch.tensor(dz).permute(0, 3, 1, 2))
    assert np.allclose(oracle.conv3x3_fwd_strided(x, w, b, 0, u=2),
                       z.detach().permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.conv3x3_dgrad_strided(dz, w, H, W, u=2),
                       xt.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)
    dw, db = oracle.conv3x3_wgrad_strided(x, dz, u=2)
    assert np.allclose(dw, wt.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# identities
# ---------------------------------------------------------------------------
def test_adjoint_identity_fwd_dgrad():
    # <fwd(x, w), v> = <x, dgrad(v, w)> with no bias and no activation
    x = rand(2, 5, 7, 3)
    w = rand(4, 3, 3, 3)
    v = rand(2, 5, 7, 4)
    lhs = np.sum(oracle.conv3x3_fwd(x, w) * v)
    rhs = np.sum(x * oracle.conv3x3_dgrad(v, w))
    assert lhs == pytest.approx(rhs, rel=1e-12)


def test_bilinear_wgrad_identity_and_dbias():
    # <dw(x, dz), V> = <fwd(x, V), dz> for any V;  db = sum of dz over pixels
    x = rand(2, 4, 6, 5)
    dz = rand(2, 4, 6, 3)
    V = rand(3, 3, 3, 5)
    dw, db = oracle.conv3x3_wgrad(x, dz)
    assert np.sum(dw * V) == pytest.approx(np.sum(oracle.conv3x3_fwd(x, V) * dz), rel=1e-12)
    assert np.allclose(db, dz.sum(axis=(0, 1, 2)), rtol=1e-13)
    assert np.allclose(oracle.conv3x3_dbias(dz), db, rtol=1e-13)


def test_wgrad_matches_central_finite_differences():
    # L(w) = <fwd(x, w), dz> is linear in w, so central differences are exact up to rounding
    x = rand(1, 4, 5, 2)
    dz = rand(1, 4, 5, 3)
    w0 = rand(3, 3, 3, 2)
    dw, _ = oracle.conv3x3_wgrad(x, dz)
    eps = 1e-3
    for e in range(w0.size):
        wp = w0.copy().reshape(-1)
        wm = w0.copy().reshape(-1)
        wp[e] += eps
        wm[e] -= eps
        lp = np.sum(oracle.conv3x3_fwd(x, wp.reshape(w0.shape)) * dz)
        lm = np.sum(oracle.conv3x3_fwd(x, wm.reshape(w0.shape)) * dz)
        assert (lp - lm) / (2 * eps) == pytest.approx(dw.reshape(-1)[e], abs=1e-9)


def test_dgrad_matches_central_finite_differences():
    x0 = rand(1, 3, 4, 2)
    w = rand(3, 3, 3, 2)
    dz = rand(1, 3, 4, 3)
    dx = oracle.conv3x3_dgrad(dz, w)
    eps = 1e-3
    for e in range(x0.size):
        xp = x0.copy().reshape(-1)
        xm = x0.copy().reshape(-1)
        xp[e] += eps
        xm[e] -= eps
        lp = np.sum(oracle.conv3x3_fwd(xp.reshape(x0.shape), w) * dz)
        lm = np.sum(oracle.conv3x3_fwd(xm.reshape(x0.shape), w) * dz)
        assert (lp - lm) / (2 * eps) == pytest.approx(dx.reshape(-1)[e], abs=1e-9)


# ---------------------------------------------------------------------------
# brute force and library special cases
# ---------------------------------------------------------------------------
def im2col(x):
    """Explicit [P, 9*Cin] patch matrix, column order (r, s, c)."""
    N, H, W, C = x.shape
    xp = np.zeros((N, H + 2, W + 2, C))
    xp[:, 1:H + 1, 1:W + 1] = x
    cols = [xp[:, r:r + H, s:s + W, :] for r in range(3) for s in range(3)]
    return np.concatenate(cols, axis=-1).reshape(N * H * W, 9 * C)


def col2im(cols, shape):
    N, H, W, C = shape
    xp = np.zeros((N, H + 2, W + 2, C))
    cols = cols.reshape(N, H, W, 9, C)
    for t in range(9):
        r, s = divmod(t, 3)
        xp[:, r:r + H, s:s + W, :] += cols[:, :, :, t, :]
    return xp[:, 1:H + 1, 1:W + 1]


def test_brute_force_im2col_all_three_passes():
    N, H, W, Cin, Cout = 2, 5, 4, 3, 6
    x = rand(N, H, W, Cin)
    w = rand(Cout, 3, 3, Cin)
    b = rand(Cout)
    dz = rand(N, H, W, Cout)
    A = im2col(x)
    Wm = w.reshape(Cout, 9 * Cin)
    y = (A @ Wm.T + b).reshape(N, H, W, Cout)
    assert np.allclose(oracle.conv3x3_fwd(x, w, b), y, rtol=1e-12, atol=1e-12)
    dx = col2im(dz.reshape(-1, Cout) @ Wm, x.shape)
    assert np.allclose(oracle.conv3x3_dgrad(dz, w), dx, rtol=1e-12, atol=1e-12)
    dw = (dz.reshape(-1, Cout).T @ A).reshape(Cout, 3, 3, Cin)
    got_dw, got_db = oracle.conv3x3_wgrad(x, dz)
    assert np.allclose(got_dw, dw, rtol=1e-12, atol=1e-12)
    assert np.allclose(got_db, dz.reshape(-1, Cout).sum(0), rtol=1e-12)


def test_torch_float64_conv2d_cross_check():
    torch = pytest.importorskip("torch")
    N, H, W, Cin, Cout = 2, 6, 5, 4, 3
    x = rand(N, H, W, Cin)
    w = rand(Cout, 3, 3, Cin)
    b = rand(Cout)
    dz = rand(N, H, W, Cout)
    xt = torch.tensor(x).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    wt = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    bt = torch.tensor(b).requires_grad_(True)
    z = torch.nn.functional.conv2d(xt, wt, bt, stride=1, padding=1)
    z.backward(torch.tensor(dz).permute(0, 3, 1, 2))
    assert np.allclose(oracle.conv3x3_fwd(x, w, b), z.detach().permute(0, 2, 3, 1).numpy(),
                       rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.conv3x3_dgrad(dz, w), xt.grad.permute(0, 2, 3, 1).numpy(),
                       rtol=1e-12, atol=1e-12)
    dw, db = oracle.conv3x3_wgrad(x, dz)
    assert np.allclose(dw, wt.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)
    ys = oracle.conv3x3_fwd(x, w, b, act=1)
    assert np.allclose(ys, torch.nn.functional.silu(z).detach().permute(0, 2, 3, 1).numpy(),
                       rtol=1e-12, atol=1e-13)
    yl = oracle.conv3x3_fwd(x, w, b, act=2)
    zl = torch.nn.functional.leaky_relu(z, negative_slope=0.2)
    assert np.allclose(yl, zl.detach().permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-13)


def test_hand_computed_fixture():
    with open(os.path.join(GOLDEN, "hand_3x3.json")) as f:
        g = json.load(f)
    x, w, b = np.array(g["x"], float), np.array(g["w"], float), np.array(g["bias"], float)
    dz = np.array(g["dz"], float)
    assert np.array_equal(oracle.conv3x3_fwd(x, w, b), np.array(g["y"], float))
    assert np.array_equal(oracle.conv3x3_dgrad(dz, w), np.array(g["dx"], float))
    dw, db = oracle.conv3x3_wgrad(x, dz)
    assert np.array_equal(dw, np.array(g["dw"], float))
    assert np.array_equal(db, np.array(g["db"], float))


# ---------------------------------------------------------------------------
# invariants and internal consistency
# ---------------------------------------------------------------------------
def test_sampled_entry_points_equal_full_results():
    N, H, W, Cin, Cout = 2, 5, 6, 3, 4
    x, w, b, dz = rand(N, H, W, Cin), rand(Cout, 3, 3, Cin), rand(Cout), rand(N, H, W, Cout)
    y = oracle.conv3x3_fwd(x, w, b, act=1)
    idx = rng.choice(y.size, 50, replace=False)
    assert np.array_equal(oracle.conv3x3_fwd_at(x, w, b, 1, idx), y.reshape(-1)[idx])
    dx = oracle.conv3x3_dgrad(dz, w)
    idx = rng.choice(dx.size, 50, replace=False)
    assert np.array_equal(oracle.conv3x3_dgrad_at(dz, w, idx), dx.reshape(-1)[idx])
    dw, _ = oracle.conv3x3_wgrad(x, dz)
    idx = rng.choice(dw.size, 50, replace=False)
    assert np.allclose(oracle.conv3x3_wgrad_at(x, dz, idx), dw.reshape(-1)[idx], rtol=1e-13, atol=1e-13)
    # the sampled dgrad through the input's activation: every element of a
    # shape whose sizes are all distinct (a slip in the index decode cannot
    # land on a value that happens to be equal), both activations
    zin = 3.0 * rand(N, H, W, Cin)
    every = np.arange(N * H * W * Cin)
    for act in (1, 2):
        full = oracle.conv3x3_dgrad_act(dz, w, zin, act)
        assert np.array_equal(oracle.conv3x3_dgrad_act_at(dz, w, zin, act, every), full.reshape(-1))
        idx = rng.choice(full.size, 50, replace=False)
        assert np.array_equal(oracle.conv3x3_dgrad_act_at(dz, w, zin, act, idx), full.reshape(-1)[idx])


def test_results_do_not_depend_on_thread_count():
    x, w, dz = rand(3, 7, 5, 4), rand(6, 3, 3, 4), rand(3, 7, 5, 6)
    try:
        oracle.set_threads(1)
        a = (oracle.conv3x3_fwd(x, w), oracle.conv3x3_dgrad(dz, w), *oracle.conv3x3_wgrad(x, dz))
        oracle.set_threads(5)
        b = (oracle.conv3x3_fwd(x, w), oracle.conv3x3_dgrad(dz, w), *oracle.conv3x3_wgrad(x, dz))
    finally:
        oracle.set_threads(0)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_stem_padding_channels_stay_exactly_zero():
    L = synth.Layer("stem-small", 2, 8, 16, 6, 5, act=1, cin_real=3)
    t = synth.make_tensors(L, seed=0)
    assert np.all(t.x[..., 3:] == 0) and np.all(t.w[..., 3:] == 0)
    dx = oracle.conv3x3_dgrad(t.dy, t.w)
    dw, _ = oracle.conv3x3_wgrad(t.x, t.dy)
    assert np.all(dx[..., 3:] == 0)
    assert np.all(dw[..., 3:] == 0)
    assert np.any(dx[..., :3] != 0) and np.any(dw[..., :3] != 0)


def test_degenerate_sizes():
    # 1x1 images: only the centre tap ever lands inside
    x, w, b = rand(3, 1, 1, 2), rand(4, 3, 3, 2), rand(4)
    y = oracle.conv3x3_fwd(x, w, b)
    assert np.allclose(y[:, 0, 0, :], x[:, 0, 0, :] @ w[:, 1, 1, :].T + b, rtol=1e-13)
    # a single row: only r = 1 taps contribute
    x, w = rand(1, 1, 6, 2), rand(3, 3, 3, 2)
    w2 = w.copy()
    w2[:, [0, 2]] = 0
    assert np.array_equal(oracle.conv3x3_fwd(x, w), oracle.conv3x3_fwd(x, w2))


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (mutated copies of the oracle, CPU only)
# ---------------------------------------------------------------------------
MUTANTS = {
    "fwd kernel flipped in h": ("int64_t hh = h + r - 1;", "int64_t hh = h - r + 1;"),
    "fwd bias dropped": ("double acc = j->bias ? j->bias[k] : 0.0;", "double acc = 0.0;"),
    "fwd weight taps transposed": ("const double* wp = j->wt + ((k * 3 + r) * 3 + s) * j->Cin;",
                                   "const double* wp = j->wt + ((k * 3 + s) * 3 + r) * j->Cin;"),
    "fwd last column of taps missing": ("for (int64_t s = 0; s < 3; ++s) {\n      int64_t ww = w + s - 1;",
                                        "for (int64_t s = 0; s < 2; ++s) {\n      int64_t ww = w + s - 1;"),
    "dgrad taps not mirrored": ("int64_t hh = h + 1 - r;", "int64_t hh = h + r - 1;"),
    "dgrad weight index off by a tap": ("acc += dzp[k] * j->wt[((k * 3 + r) * 3 + s) * j->Cin + c];",
                                        "acc += dzp[k] * j->wt[((k * 3 + s) * 3 + r) * j->Cin + c];"),
    "wgrad shifted the wrong way": ("            int64_t ww = w + s - 1;\n            if (ww < 0 || ww >= j->W) continue;\n            const double* xp",
                                    "            int64_t ww = w - s + 1;\n            if (ww < 0 || ww >= j->W) continue;\n            const double* xp"),
    "dbias squares dz": ("db += d;", "db += d * d;"),
    "silu sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "leaky relu slope": ("return z >= 0.0 ? z : 0.2 * z;", "return z >= 0.0 ? z : 0.02 * z;"),
    "leaky relu on the wrong side": ("return z >= 0.0 ? z : 0.2 * z;", "return z >= 0.0 ? 0.2 * z : z;"),
    "leaky relu not applied": ("if (act == 2) return oracle_lrelu_f64(z);", "if (act == 2) return z;"),
    "silu grad without the (1 - s) factor": ("return sg * (1.0 + z * (1.0 - sg));", "return sg * (1.0 + z);"),
    "leaky relu grad slope": ("return z > 0.0 ? 1.0 : 0.2;", "return z > 0.0 ? 1.0 : 0.02;"),
    "strided forward ignores the row stride": ("    int64_t hh = j->u * ho + r - 1;", "    int64_t hh = ho + r - 1;"),
    "strided dgrad skips the parity test": ("if (th < 0 || th % j->u != 0 || th / j->u >= Ho) continue;",
                                            "if (th < 0 || th / j->u >= Ho) continue;"),
    "strided wgrad column off by one": ("        int64_t ww = j->u * wo + s - 1;", "        int64_t ww = j->u * wo + s;"),
    "strided dbias drops the last image": ("for (int64_t p = 0; p < j->N * Ho * Wo; ++p)",
                                           "for (int64_t p = 0; p < (j->N - 1) * Ho * Wo; ++p)"),
    "sampled dgrad_act reads zin at the pixel, not the element": (
        "j->out[i] = oracle_act_grad_f64(j->act, j->zin[e])", "j->out[i] = oracle_act_grad_f64(j->act, j->zin[p])"),
    "sampled dgrad_act decodes the row one off": (
        "int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);\n  j->out[i] = oracle_act_grad_f64",
        "int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);\n  h = (h + 1) % j->H;\n"
        "  j->out[i] = oracle_act_grad_f64"),
    "sampled wgrad decodes the tap transposed": ("int64_t r = rs / 3, s = rs % 3;", "int64_t r = rs % 3, s = rs / 3;"),
    "dgrad_act reads zin of channel 0": ("j->out[e] = oracle_act_grad_f64(j->act, j->zin[e]) * dgrad_point(j, n, h, w, c);",
                                         "j->out[e] = oracle_act_grad_f64(j->act, j->zin[e - c]) * dgrad_point(j, n, h, w, c);"),
}


def _mutant_module(tmp_path, name, old, new):
    import importlib.util
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    d = tmp_path / name.replace(" ", "_")
    d.mkdir()
    (d / "conv3x3_oracle.c").write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("oracle_mutant", oracle.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "conv3x3_oracle.c")
    mod._LIB = str(d / "liboracle.so")
    mod._lib = None
    return mod


def _suite():
    return [
        test_centre_delta_reproduces_input,
        *[(lambda r=r, s=s: test_off_centre_delta_shifts_with_zero_fill(r, s))
          for r in range(3) for s in range(3)],
        test_all_ones_kernel_on_constant_input_gives_9_6_4_pattern,
        test_one_by_one_special_case_is_a_gemm,
        test_silu_special_values_and_grid,
        test_leaky_relu_special_values_and_epilogue,
        test_act_grad_closed_forms_and_finite_differences,
        test_strided_with_stride_one_is_the_plain_convolution,
        (lambda: test_stride_two_forward_is_the_plain_output_at_even_positions(7, 5)),
        (lambda: test_stride_two_backward_identities(7, 5)),
        (lambda: test_dgrad_through_activation_by_finite_differences(1)),
        (lambda: test_dgrad_through_activation_by_finite_differences(2)),
        test_adjoint_identity_fwd_dgrad,
        test_bilinear_wgrad_identity_and_dbias,
        test_brute_force_im2col_all_three_passes,
        test_hand_computed_fixture,
        test_sampled_entry_points_equal_full_results,
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(tmp_path, name):
    old, new = MUTANTS[name]
    mod = _mutant_module(tmp_path, name, old, new)
    g = globals()
    saved = g["oracle"]
    g["oracle"] = mod
    caught = 0
    try:
        for fn in _suite():
            try:
                fn()
            except AssertionError:
                caught += 1
    finally:
        g["oracle"] = saved
    assert caught > 0, "no pin caught the planted mistake: " + name
