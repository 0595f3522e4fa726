"""Pins of the upfirdn2d oracle (CPU only): it is checked against things other
than itself -- hand-worked cases, library routines it reduces to, closed forms
and identities of the operation -- and each planted mistake in a mutated copy
of its source is caught by at least one pin.

The operation (StyleGAN2 custom-kernel blog, page titled "Dim3 grid
calculation code", first paragraph): upsample by inserting zeros after each
pixel, pad with zeros, FIR-filter by convolution, downsample by dropping
pixels; every channel of every image on its own.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
rng = np.random.default_rng(2024)


def rand(*shape):
    return rng.standard_normal(shape)


def binomial4():
    a = np.array([1.0, 3.0, 3.0, 1.0])
    return np.outer(a, a) / 64.0


def test_hand_worked_cases():
    with open(os.path.join(GOLDEN, "upfirdn2d_hand.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        y = oracle.upfirdn2d(np.array(c["x"], float), np.array(c["f"], float), c["up"], c["down"],
                             c["pad"])
        assert np.array_equal(y, np.array(c["y"], float)), c["what"]


def test_unit_filter_without_resampling_is_the_identity():
    x = rand(2, 5, 7, 3)
    assert np.array_equal(oracle.upfirdn2d(x, np.ones((1, 1)), 1, 1, 0), x)
    # a centred delta with one pixel of zero padding on every side, too
    d = np.zeros((3, 3))
    d[1, 1] = 1.0
    assert np.array_equal(oracle.upfirdn2d(x, d, 1, 1, 1), x)


def test_plain_filter_is_scipy_convolve2d():
    sig = pytest.importorskip("scipy.signal")
    x, f = rand(2, 6, 9, 3), rand(3, 4)
    # zero pad (x0, x1, y0, y1) then the 'valid' 2-D convolution
    pad = (2, 1, 1, 1)
    y = oracle.upfirdn2d(x, f, 1, 1, pad)
    for n in range(2):
        for c in range(3):
            xp = np.pad(x[n, :, :, c], ((pad[2], pad[3]), (pad[0], pad[1])))
            ref = sig.convolve2d(xp, f, mode="valid")
            assert np.allclose(y[n, :, :, c], ref, rtol=1e-12, atol=1e-12)


def _one_axis(v, f1, up, down, p0, p1):
    """The four steps along one axis of a 1-D signal, with numpy's convolve."""
    u = np.zeros(len(v) * up)
    u[::up] = v
    pd = np.concatenate([np.zeros(p0), u, np.zeros(p1)])
    return np.convolve(pd, f1, mode="valid")[::down]


@pytest.mark.parametrize("up,down", [(1, 1), (2, 1), (1, 2), (2, 2), (3, 2)])
def test_separable_filter_is_two_one_dimensional_passes(up, down):
    x = rand(2, 5, 6, 2)
    fy, fx = rand(4), rand(3)
    pad = (2, 1, 1, 3)
    y = oracle.upfirdn2d(x, np.outer(fy, fx), up, down, pad)
    for n in range(2):
        for c in range(2):
            rows = np.array([_one_axis(r, fx, up, down, pad[0], pad[1]) for r in x[n, :, :, c]])
            ref = np.array([_one_axis(col, fy, up, down, pad[2], pad[3]) for col in rows.T]).T
            assert ref.shape == y.shape[1:3]
            assert np.allclose(y[n, :, :, c], ref, rtol=1e-12, atol=1e-12)


def test_nearest_neighbour_and_decimation_closed_forms():
    x = rand(2, 4, 5, 3)
    # box filter after 2x upsampling, pad before: every pixel repeated 2x2
    y = oracle.upfirdn2d(x, np.ones((2, 2)), 2, 1, (1, 0, 1, 0))
    assert np.array_equal(y, np.repeat(np.repeat(x, 2, axis=1), 2, axis=2))
    # unit filter and 2x downsampling: the even pixels (odd and even sizes)
    z = rand(2, 9, 8, 3)
    assert np.array_equal(oracle.upfirdn2d(z, np.ones((1, 1)), 1, 2, 0), z[:, ::2, ::2, :])


def test_normalised_filter_keeps_a_constant_interior():
    c = 1.75
    x = np.full((1, 8, 8, 2), c)
    f = binomial4()
    # 2x up (filter gain 4 = up^2) and 2x down, StyleGAN2-style pads
    yu = oracle.upfirdn2d(x, 4.0 * f, 2, 1, (2, 1, 2, 1))
    assert yu.shape == (1, 16, 16, 2)
    assert np.allclose(yu[:, 2:-2, 2:-2, :], c, rtol=1e-14)
    yd = oracle.upfirdn2d(x, f, 1, 2, (1, 1, 1, 1))
    assert yd.shape == (1, 4, 4, 2)
    assert np.allclose(yd[:, 1:-1, 1:-1, :], c, rtol=1e-14)
    # and the border rows are smaller (zeros enter through the padding)
    assert np.all(yd[:, 0, :, :] < c)


@pytest.mark.parametrize("up,down,kh,kw,pad", [(2, 1, 4, 4, (2, 1, 2, 1)), (1, 2, 4, 4, (1, 1, 1, 1)),
                                               (2, 2, 3, 5, (1, 2, 2, 0)), (3, 1, 2, 3, (0, 2, 1, 1))])
def test_adjoint_swaps_up_and_down_and_flips_the_filter(up, down, kh, kw, pad):
    # <A x, v> = <x, B v> with A = upfirdn(up, down, f, pads) and
    # B = upfirdn(down, up, f flipped, pads p0' = k - 1 - p0, p1' closing the size)
    N, H, W, C = 2, 6, 5, 3
    x, f = rand(N, H, W, C), rand(kh, kw)
    px0, px1, py0, py1 = pad
    y = oracle.upfirdn2d(x, f, up, down, pad)
    Ho, Wo = y.shape[1:3]
    v = rand(N, Ho, Wo, C)
    # the far pads only have to be long enough for B's output to reach the
    # input's size; positions past the last one B reads never matter
    qx0, qy0 = kw - 1 - px0, kh - 1 - py0
    qx1 = max((W - 1) * up + kw - qx0 - Wo * down, 0)
    qy1 = max((H - 1) * up + kh - qy0 - Ho * down, 0)
    assert min(qx0, qy0) >= 0
    bv = oracle.upfirdn2d(v, f[::-1, ::-1], down, up, (qx0, qx1, qy0, qy1))
    assert bv.shape == x.shape
    lhs, rhs = np.sum(y * v), np.sum(x * bv)
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0)


def test_output_size_formula():
    for (L, up, down, p0, p1, k, want) in [(64, 2, 1, 2, 1, 4, 128), (64, 1, 2, 1, 1, 4, 32),
                                           (7, 1, 2, 1, 1, 4, 3), (5, 3, 2, 0, 0, 2, 7)]:
        assert oracle.upfirdn2d_out_len(L, up, down, p0, p1, k) == want
        x = np.zeros((1, L, 1, 1))
        assert oracle.upfirdn2d(x, np.ones((k, 1)), up, down, (0, 0, p0, p1)).shape[1] == want


@pytest.mark.parametrize("up,down,pad", [(2, 1, (2, 1, 2, 1)), (1, 2, (1, 1, 1, 1)), (2, 2, (1, 2, 0, 3))])
def test_sampled_entry_point_equals_the_full_result(up, down, pad):
    x, f = rand(2, 5, 7, 3), rand(4, 3)
    y = oracle.upfirdn2d(x, f, up, down, pad)
    every = np.arange(y.size)
    assert np.allclose(oracle.upfirdn2d_at(x, f, up, down, pad, every), y.reshape(-1),
                       rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (mutated copies of the oracle, CPU only)
# ---------------------------------------------------------------------------
MUTANTS = {
    "zeros inserted before each pixel": (
        "u[(h * j->up) * Wu + w * j->up] =", "u[(h * j->up + j->up - 1) * Wu + w * j->up + j->up - 1] ="),
    "filter not flipped (a correlation)": (
        "pd[(m + j->kh - 1 - a) * Wp + (l + j->kw - 1 - b)]", "pd[(m + a) * Wp + (l + b)]"),
    "padding placed on the far side of each axis": (
        "pd[(h + j->py0) * Wp + (w + j->px0)] = u[h * Wu + w];", "pd[(h + j->py1) * Wp + (w + j->px1)] = u[h * Wu + w];"),
    "columns not downsampled": (
        "fl[(oh * j->down) * Wf + ow * j->down]", "fl[(oh * j->down) * Wf + ow]"),
    "filter rows and columns transposed": (
        "acc += j->f[a * j->kw + b] * pd[", "acc += j->f[b * j->kh + a] * pd["),
    "sampled form ignores the upsampling phase": (
        "if (ru < 0 || ru >= j->H * j->up || ru % j->up != 0) continue;", "if (ru < 0 || ru >= j->H * j->up) continue;"),
    "sampled form drops the column padding": (
        "const int64_t cu = ow * j->down + j->kw - 1 - b - j->px0;", "const int64_t cu = ow * j->down + j->kw - 1 - b;"),
}


def _mutant_module(tmp_path, name, old, new):
    import importlib.util
    src = open(oracle._SRC_UFD).read()
    assert src.count(old) == 1, name
    d = tmp_path / name.replace(" ", "_").replace("(", "").replace(")", "")
    d.mkdir()
    (d / "upfirdn2d_oracle.c").write_text(src.replace(old, new, 1))
    (d / "conv3x3_oracle.c").write_text(open(oracle._SRC).read())
    spec = importlib.util.spec_from_file_location("oracle_mutant_ufd", oracle.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "conv3x3_oracle.c")
    mod._SRC_UFD = str(d / "upfirdn2d_oracle.c")
    mod._LIB = str(d / "liboracle.so")
    mod._lib = None
    return mod


def _suite():
    return [
        test_hand_worked_cases,
        test_unit_filter_without_resampling_is_the_identity,
        test_plain_filter_is_scipy_convolve2d,
        *[(lambda u=u, d=d: test_separable_filter_is_two_one_dimensional_passes(u, d))
          for u, d in [(1, 1), (2, 1), (1, 2), (2, 2), (3, 2)]],
        test_nearest_neighbour_and_decimation_closed_forms,
        test_normalised_filter_keeps_a_constant_interior,
        (lambda: test_adjoint_swaps_up_and_down_and_flips_the_filter(2, 2, 3, 5, (1, 2, 2, 0))),
        test_output_size_formula,
        *[(lambda u=u, d=d, p=p: test_sampled_entry_point_equals_the_full_result(u, d, p))
          for u, d, p in [(2, 1, (2, 1, 2, 1)), (1, 2, (1, 1, 1, 1)), (2, 2, (1, 2, 0, 3))]],
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
            except (AssertionError, ValueError):
                caught += 1
    finally:
        g["oracle"] = saved
    assert caught > 0, "no pin caught the planted mistake: " + name
