"""GPU parity of upfirdn2d (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs.

Tolerances (max|err| / max|ref| per output tensor):
  * fp32 result (out_dtype F32) ........................... <= 1e-5: at most
    64 fp32 products of bf16-exact inputs and fp32 taps, summed in fp32
  * bf16-stored y: elementwise |y - ref| <= ulp_bf16(ref)/2 + 1e-5 max|ref| and
    bit-identical to round-to-nearest-even of the fp32 result (one rounding)
The oracle gets the taps as the kernel sees them (rounded to fp32).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from x3_convolution_gb300 import _lib as L
from x3_convolution_gb300 import ops

from gpu_util import check_bf16_store, host, rel_err, rne_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    L.load()
    yield
    torch.cuda.synchronize()


def _case(N, C, H, W, kh, kw, seed):
    x = synth.bf16_round(synth.normal(synth.stream_id(seed, 200, 0), (N, H, W, C)))
    f = synth.normal(synth.stream_id(seed, 200, 1), (kh, kw)).astype(np.float32)
    return x, f


CASES = [
    # N, C, H, W, up, down, (px0, px1, py0, py1), kh, kw
    (2, 64, 16, 16, 2, 1, (2, 1, 2, 1), 4, 4),     # 2x up, binomial-sized
    (2, 64, 16, 16, 1, 2, (1, 1, 1, 1), 4, 4),     # 2x down
    (1, 128, 9, 7, 2, 1, (2, 1, 2, 1), 4, 4),      # odd sizes
    (1, 8, 11, 13, 1, 2, (1, 2, 0, 3), 4, 3),      # C = 8, asymmetric pads, odd output
    (3, 24, 5, 6, 1, 1, (1, 1, 1, 1), 3, 3),       # plain FIR
    (2, 16, 6, 5, 3, 2, (2, 0, 1, 3), 5, 2),       # generic factors (run-time up / down)
    (1, 32, 4, 4, 4, 1, (3, 3, 3, 3), 8, 8),       # largest taps, 4x up
    (1, 40, 1, 1, 2, 1, (2, 1, 2, 1), 4, 4),       # 1x1 image
    (2, 16, 7, 9, 2, 2, (0, 0, 0, 0), 1, 1),       # unit filter: decimated zero-insertion
    (1, 512, 8, 8, 2, 1, (2, 1, 2, 1), 4, 4),      # many channel groups per pixel
    (1, 16, 5, 5, 1, 1, (9, 0, 0, 9), 2, 2),       # pads wider than the image
    # the 2x up / 2x down 4x4 kernels with every pad parity and odd output sizes
    (1, 16, 5, 6, 2, 1, (1, 2, 3, 0), 4, 4),       # first output block starts at row / column 0
    (2, 8, 3, 4, 2, 1, (4, 3, 0, 5), 4, 4),
    (2, 24, 7, 9, 1, 2, (0, 3, 2, 1), 4, 4),
    (1, 8, 1, 1, 1, 2, (2, 1, 1, 2), 4, 4),        # 1x1 input, output 1x1
    (1, 64, 6, 11, 1, 2, (3, 0, 0, 3), 4, 4),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + "_k%dx%d" % c[7:9])
def test_small_cases_full_tensors(case):
    N, C, H, W, up, down, pad, kh, kw = case
    x, f = _case(N, C, H, W, kh, kw, seed=len(str(case)))
    xd = to_dev_bf16(x)
    y32 = ops.upfirdn2d(xd, f, up, down, pad, out_dtype=L.DT_F32)
    ybf = ops.upfirdn2d(xd, f, up, down, pad)
    torch.cuda.synchronize()
    ref = oracle.upfirdn2d(x, f.astype(np.float64), up, down, pad)
    assert y32.shape == ref.shape
    assert rel_err(host(y32), ref) <= TOL
    assert check_bf16_store(host(ybf), ref, tol=TOL) == 0
    assert np.array_equal(host(ybf), rne_bf16(host(y32)))


def test_adjoint_pair_on_the_gpu():
    # the input gradient of a 2x upsampling is a 2x downsampling with the
    # flipped filter: <up(x), v> = <x, down(v)> in the kernel's own arithmetic
    N, C, H, W = 2, 64, 8, 8
    x, _ = _case(N, C, H, W, 4, 4, seed=3)
    f = synth.Resample("u", N, C, H, W, up=2, pad=(2, 1, 2, 1)).filter()
    y = ops.upfirdn2d(to_dev_bf16(x), f, 2, 1, (2, 1, 2, 1), out_dtype=L.DT_F32)
    v = synth.bf16_round(synth.normal(synth.stream_id(3, 201, 0), tuple(y.shape)))
    # leading pads k - 1 - p0 = 1, trailing pads closing the size: (W-1)*2 + 4 - 1 - 2W = 1
    bv = ops.upfirdn2d(to_dev_bf16(v), f[::-1, ::-1].copy(), 1, 2, (1, 1, 1, 1), out_dtype=L.DT_F32)
    torch.cuda.synchronize()
    assert tuple(bv.shape) == (N, H, W, C)
    lhs = float(np.sum(host(y) * v))
    rhs = float(np.sum(x * host(bv)))
    assert abs(lhs - rhs) <= 1e-5 * max(abs(lhs), 1.0)


@pytest.mark.parametrize("index", range(len(synth.UPFIRDN2D)))
def test_unet_resampling_full_size_sampled(index):
    # the benchmark's ops at batch 64: random outputs plus every output of the
    # first and last image (all borders), against the oracle one by one
    op = synth.UPFIRDN2D[index]
    x = synth.make_resample_input(op, seed=0, index=index)
    f = op.filter()
    xd = to_dev_bf16(x)
    y32 = ops.upfirdn2d(xd, f, op.up, op.down, op.pad, out_dtype=L.DT_F32)
    ybf = ops.upfirdn2d(xd, f, op.up, op.down, op.pad)
    torch.cuda.synchronize()
    y32h, ybfh = host(y32).reshape(-1), host(ybf).reshape(-1)
    per_img = op.Ho * op.Wo * op.C
    rng = np.random.default_rng(300 + index)
    idx = np.concatenate([rng.integers(0, y32h.size, 8192), np.arange(per_img),
                          np.arange(y32h.size - per_img, y32h.size)])
    ref = oracle.upfirdn2d_at(x, f.astype(np.float64), op.up, op.down, op.pad, idx)
    assert np.max(np.abs(y32h[idx] - ref)) / max(np.max(np.abs(ref)), 1e-30) <= TOL
    assert np.array_equal(ybfh[idx], rne_bf16(y32h[idx]))


def test_bad_arguments_raise():
    x = torch.zeros((1, 8, 8, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.Conv3x3Error) as e:
        ops.upfirdn2d(x, np.ones((4, 4), np.float32), 2, 1, (2, 1, 2, 1))
    assert e.value.status == L.ERR_INVALID_ARG
