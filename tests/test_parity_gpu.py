"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs.

Tolerances (max|err| / max|ref| per output tensor):
  * fp32 check path, all tensors fp32 ............................ <= 1e-5
  * bf16 inputs, fp32 accumulation, fp32 result (out_dtype=F32) ... <= 2e-3
  * bf16-stored y / dx: elementwise |y - ref| <= ulp_bf16(ref)/2 + 2e-3 max|ref|
    and bit-identical to round-to-nearest-even of the fp32 result of the same
    kernel (one rounding, on store)
  * dw, dbias (fp32 outputs) ..................................... <= 2e-3
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from x3_convolution_gb300 import _lib as L
from x3_convolution_gb300 import ops

from gpu_util import check_bf16_store, host, rel_err, rne_bf16, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-3
TOL_F32 = 1e-5
PATHS = {"tensor": L.PATH_TENSOR, "simt": L.PATH_SIMT}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    L.load()
    yield
    torch.cuda.synchronize()
    assert L.conv3x3_device_status() == L.OK


def dev_tensors(t):
    return (to_dev_bf16(t.x), to_dev_bf16(t.w), to_dev_f32(t.bias), to_dev_bf16(t.dy))


# ---------------------------------------------------------------------------
# fp32 check path: the tiny workload, full tensors
# ---------------------------------------------------------------------------
def test_tiny_fp32_check_path_full():
    Lr = synth.TINY
    t = synth.make_tensors(Lr, seed=0)
    x, w, b, dy = (to_dev_f32(a) for a in (t.x, t.w, t.bias, t.dy))
    y = ops.fwd_f32(x, w, b, act=L.ACT_NONE)
    dx = ops.dgrad_f32(dy, w)
    dw, db = ops.wgrad_f32(x, dy)
    torch.cuda.synchronize()
    assert rel_err(host(y), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) <= TOL_F32
    assert rel_err(host(dx), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_F32
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_F32
    assert rel_err(host(db), rdb) <= TOL_F32
    ys = ops.fwd_f32(x, w, b, act=L.ACT_SILU)
    assert rel_err(host(ys), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) <= TOL_F32
    yl = ops.fwd_f32(x, w, b, act=L.ACT_LRELU)
    assert rel_err(host(yl), oracle.conv3x3_fwd(t.x, t.w, t.bias, 2)) <= TOL_F32


def test_tiny_in_bf16_at_the_bf16_gate():
    Lr = synth.Layer("tiny-bf16", 2, 64, 64, 32, 32, act=0)
    t = synth.make_tensors(Lr, seed=0)
    x, w, b, dy = dev_tensors(t)
    y = ops.fwd(x, w, b, act=0, out_dtype=L.DT_F32)
    dx = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    dw, db = ops.wgrad(x, dy)
    torch.cuda.synchronize()
    assert rel_err(host(y), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) <= TOL_BF16
    assert rel_err(host(dx), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16


# ---------------------------------------------------------------------------
# small shapes, full tensors: several tiles, ragged tails, edge cases, both paths
# ---------------------------------------------------------------------------
SHAPES = [
    # N, Cin, Cout, H, W
    (2, 64, 64, 9, 9),        # P = 162: two 128-pixel tiles, ragged tail
    (1, 128, 128, 16, 16),    # exact tiles
    (3, 64, 192, 5, 7),       # P < 128, tiles cross image boundaries, N tile 192
    (2, 256, 256, 8, 8),      # N tile 256, K = 2304
    (1, 72, 200, 6, 11),      # ragged channel chunk (72) and ragged N tile (200)
    (2, 8, 128, 12, 12),      # stem-like Cin = 8
    (1, 16, 24, 3, 5),        # tiny channel counts
    (1, 64, 64, 1, 1),        # 1x1 images: only the centre tap lands
    (2, 64, 64, 2, 3),        # H, W in {2, 3}
    (1, 384, 128, 4, 4),      # Cin 384 (6 chunks), dgrad N tile 384 -> 192
    (5, 128, 64, 1, 37),      # single-row images
    (1, 64, 512, 3, 3),       # Cout 512: two N tiles of 256
]


def _small(shape, act=1, seed=7):
    N, Cin, Cout, H, W = shape
    Lr = synth.Layer("s", N, Cin, Cout, H, W, act=act)
    return synth.make_tensors(Lr, seed=seed)


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_all_passes(shape, path):
    p = PATHS[path]
    t = _small(shape)
    x, w, b, dy = dev_tensors(t)
    for act in (0, 1, 2):
        y32 = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=p)
        ybf = ops.fwd(x, w, b, act=act, out_dtype=L.DT_BF16, path=p)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_fwd(t.x, t.w, t.bias, act)
        assert rel_err(host(y32), ref) <= TOL_BF16, ("fwd", act)
        assert check_bf16_store(host(ybf), ref) == 0, ("fwd bf16 store", act)
        assert np.array_equal(host(ybf), rne_bf16(host(y32))), ("fwd one rounding", act)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p)
    dxbf = ops.dgrad(dy, w, out_dtype=L.DT_BF16, path=p)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_dgrad(t.dy, t.w)
    assert rel_err(host(dx32), ref) <= TOL_BF16
    assert check_bf16_store(host(dxbf), ref) == 0
    assert np.array_equal(host(dxbf), rne_bf16(host(dx32)))
    dw, db = ops.wgrad(x, dy, path=p)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16


# "128x2" runs transposed (channels on TMEM lanes), "128x2n" is the same tile untransposed;
# "256x1" runs on two-CTA clusters (one 256-pixel x 256-channel tile per pair), "256x1n" on
# one CTA; "pair<BN>" runs 256-pixel x BN-channel tiles on two-CTA clusters
TILES = ["64x1", "128x1", "192x1", "256x1", "256x1n", "64x2", "128x2", "128x2n",
         "pair128", "pair192", "pair256", "pair384"]


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("shape", [(2, 64, 64, 9, 9), (1, 72, 200, 6, 11), (3, 128, 256, 17, 13),
                                   (2, 8, 128, 12, 12)], ids=lambda s: "x".join(map(str, s)))
def test_every_tensor_tile_shape(shape, tile, monkeypatch):
    monkeypatch.setenv("CONV3X3_TILE", tile)
    t = _small(shape)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) <= TOL_BF16
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16


@pytest.mark.parametrize("kc", ["2", "1"], ids=["two_chunks", "one_chunk"])
@pytest.mark.parametrize("shape", [(1, 72, 200, 6, 11), (2, 256, 256, 8, 8), (1, 192, 320, 5, 7)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_chunks_per_stage(shape, kc, monkeypatch):
    # CTA-pair tiles with one or two 64-channel chunks per stage (two only where
    # the chunk count is even: 192 input channels keep one in the forward)
    monkeypatch.setenv("CONV3X3_TILE", "pair256")
    monkeypatch.setenv("CONV3X3_PAIR_KC", kc)
    t = _small(shape, seed=37)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) <= TOL_BF16
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16


@pytest.mark.parametrize("kc", ["2", "1"], ids=["two_chunks", "one_chunk"])
@pytest.mark.parametrize("shape", [(1, 72, 200, 6, 11), (2, 256, 256, 8, 8), (3, 128, 256, 17, 13)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_half_width_items(shape, kc, monkeypatch):
    # every 256-channel pair tile as two 128-channel items (N = 128 MMAs over
    # 64 weight rows per CTA): plain, bf16 through TMA stores, the forward's
    # z store and the dgrad's z_in scaling; 200 and 72 output channels leave
    # the second item partly or wholly past the last channel
    monkeypatch.setenv("CONV3X3_TILE", "pair256")
    monkeypatch.setenv("CONV3X3_PAIR_KC", kc)
    monkeypatch.setenv("CONV3X3_PAIR_HALF", "all")
    t = _small(shape, seed=43)
    x, w, b, dy = dev_tensors(t)
    zin_h = synth.make_zin(t.layer, seed=43)
    N, Cin, Cout, H, W = shape
    z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    ybf = ops.fwd(x, w, b, act=1, path=L.PATH_TENSOR)
    ops.fwd(x, w, b, act=1, path=L.PATH_TENSOR, z_out=z)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    gx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR, z_in=to_dev_bf16(zin_h), act_in=1)
    torch.cuda.synchronize()
    ry = oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)
    assert rel_err(host(y32), ry) <= TOL_BF16
    assert check_bf16_store(host(ybf), ry) == 0
    assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) == 0
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16
    assert rel_err(host(gx32), oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)) <= TOL_BF16


def test_pair_last_round_half_width_full_size(monkeypatch):
    # 256 -> 256 channels at 32x32, batch 64: 256 pair tiles over the pairs
    # that fit (76 on a 152-SM GPU) leave a last round of 28 tiles, which runs
    # as 56 half-width items; against whole tiles and the oracle's last pixels
    Lr = synth.L2
    t = synth.make_tensors(Lr, seed=5)
    x, w, b, dy = dev_tensors(t)
    y = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32)
    dx = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    monkeypatch.setenv("CONV3X3_PAIR_HALF", "0")
    y0 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32)
    dx0 = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    torch.cuda.synchronize()
    assert rel_err(host(y), host(y0)) <= 1e-6
    assert rel_err(host(dx), host(dx0)) <= 1e-6
    P = Lr.N * Lr.H * Lr.W
    pix = np.array([P - 7 * 256 - 1, P - 256, P - 129, P - 1])
    iy = (pix[:, None] * Lr.Cout + np.arange(Lr.Cout)[None, :]).reshape(-1)
    ix = (pix[:, None] * Lr.Cin + np.arange(Lr.Cin)[None, :]).reshape(-1)
    ry = oracle.conv3x3_fwd_at(t.x, t.w, t.bias, 1, iy)
    rx = oracle.conv3x3_dgrad_at(t.dy, t.w, ix)
    assert np.max(np.abs(host(y).reshape(-1)[iy] - ry)) / np.max(np.abs(ry)) <= TOL_BF16
    assert np.max(np.abs(host(dx).reshape(-1)[ix] - rx)) / np.max(np.abs(rx)) <= TOL_BF16


PKS_SHAPES = [
    # N, Cin, Cout, H, W: one 256 x 256 tile per cluster of four, K split over its two pairs
    (2, 256, 256, 8, 8),      # one tile, the second CTA of each pair past the last pixel
    (4, 512, 512, 8, 8),      # two tiles across the output channels
    (5, 256, 512, 10, 11),    # six tiles, ragged pixel tail
    (2, 384, 256, 9, 9),      # 27 k-blocks: halves of 14 and 13 (dgrad: 384 outputs, other tiles)
]


@pytest.mark.parametrize("shape", PKS_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_tiles_with_k_split_over_two_pairs(shape, monkeypatch):
    monkeypatch.setenv("CONV3X3_PKS", "1")
    t = _small(shape, seed=47)
    x, w, b, dy = dev_tensors(t)
    zin_h = synth.make_zin(t.layer, seed=47)
    N, Cin, Cout, H, W = shape
    z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    ybf = ops.fwd(x, w, b, act=1, path=L.PATH_TENSOR, z_out=z)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    gx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR, z_in=to_dev_bf16(zin_h), act_in=1)
    y32b = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert torch.equal(y32, y32b)  # the two K halves are added in a fixed way
    ry = oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)
    assert rel_err(host(y32), ry) <= TOL_BF16
    assert check_bf16_store(host(ybf), ry) == 0
    assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) == 0
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16
    assert rel_err(host(gx32), oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)) <= TOL_BF16


def test_pair_k_split_8x8_layer_full_size(monkeypatch):
    # 512 -> 512 channels at 8x8, batch 64 (32 tiles, 128 CTAs), the AUTO path,
    # against one-CTA tiles and the oracle's first and last pixels
    Lr = synth.Layer("pks", 64, 512, 512, 8, 8, act=1)
    t = synth.make_tensors(Lr, seed=9)
    x, w, b, dy = dev_tensors(t)
    y = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32)
    dx = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    monkeypatch.setenv("CONV3X3_PKS", "0")
    y0 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32)
    dx0 = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    torch.cuda.synchronize()
    assert rel_err(host(y), host(y0)) <= 1e-5
    assert rel_err(host(dx), host(dx0)) <= 1e-5
    P = Lr.N * Lr.H * Lr.W
    pix = np.array([0, 1, 129, 255, 256, P - 257, P - 1])
    iy = (pix[:, None] * Lr.Cout + np.arange(Lr.Cout)[None, :]).reshape(-1)
    ix = (pix[:, None] * Lr.Cin + np.arange(Lr.Cin)[None, :]).reshape(-1)
    ry = oracle.conv3x3_fwd_at(t.x, t.w, t.bias, 1, iy)
    rx = oracle.conv3x3_dgrad_at(t.dy, t.w, ix)
    assert np.max(np.abs(host(y).reshape(-1)[iy] - ry)) / np.max(np.abs(ry)) <= TOL_BF16
    assert np.max(np.abs(host(dx).reshape(-1)[ix] - rx)) / np.max(np.abs(rx)) <= TOL_BF16


@pytest.mark.parametrize("pair384", ["auto", "0"], ids=["pair384", "one_cta"])
@pytest.mark.parametrize("shape", [(2, 384, 384, 16, 16), (1, 256, 384, 16, 16), (3, 128, 384, 9, 13),
                                   (1, 896, 384, 8, 8)], ids=lambda s: "x".join(map(str, s)))
def test_384_channel_tiles(shape, pair384, monkeypatch):
    # 256 x 384 two-CTA tiles (which the full-size 16x16 layers take by
    # default; forced here) against the one-CTA tiles
    if pair384 == "0":
        monkeypatch.setenv("CONV3X3_PAIR384", "0")
    else:
        monkeypatch.setenv("CONV3X3_TILE", "pair384")
    t = _small(shape, seed=41)
    x, w, b, dy = dev_tensors(t)
    for act in (1, 2):
        y32 = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
        ybf = ops.fwd(x, w, b, act=act, path=L.PATH_TENSOR)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_fwd(t.x, t.w, t.bias, act)
        assert rel_err(host(y32), ref) <= TOL_BF16
        assert np.array_equal(host(ybf), rne_bf16(host(y32)))
    # dgrad: 384 outputs where Cin = 384
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16


KSPLIT_SHAPES = [
    # N, Cin, Cout, H, W: 256-channel output tiles whose K is split over a CTA pair
    (2, 128, 256, 8, 8),
    (1, 72, 512, 5, 7),      # ragged chunk, ragged pixel tail, two channel tiles
    (3, 512, 256, 8, 8),     # long K
    (1, 64, 256, 3, 3),      # nine k-blocks: five and four per CTA
]


@pytest.mark.parametrize("ks", ["1", "0"], ids=["ksplit", "plain"])
@pytest.mark.parametrize("shape", KSPLIT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_k_split_tiles(shape, ks, monkeypatch):
    monkeypatch.setenv("CONV3X3_KSPLIT", ks)
    t = _small(shape, seed=43)
    x, w, b, dy = dev_tensors(t)
    for act in (1, 2):
        y32 = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
        ybf = ops.fwd(x, w, b, act=act, path=L.PATH_TENSOR)
        y32b = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
        torch.cuda.synchronize()
        assert rel_err(host(y32), oracle.conv3x3_fwd(t.x, t.w, t.bias, act)) <= TOL_BF16
        assert np.array_equal(host(ybf), rne_bf16(host(y32)))
        assert torch.equal(y32, y32b)  # the cross-CTA sum is deterministic
    # dgrad needs Cin a multiple of 256 for this tile; the others take the plain kernels
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16


def test_k_split_fused_and_concat(monkeypatch):
    # the fused activation backward and the concat-free calls on K-split tiles
    monkeypatch.setenv("CONV3X3_KSPLIT", "1")
    shape = (2, 192, 64, 256, 6, 7)  # N, Ca, Cb, Cout, H, W: a chunk pair across the split
    N, Ca, Cb, Cout, H, W = shape
    t, zin_h, _ = _cat_case(shape)
    x, w, b, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    y32 = ops.fwd_cat(xa, xb, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd_cat(t.x[..., :Ca], t.x[..., Ca:], t.w, t.bias, 1)) <= TOL_BF16
    zin = to_dev_bf16(zin_h)
    za, zb = zin[..., :Ca].contiguous(), zin[..., Ca:].contiguous()
    gxa, gxb = ops.dgrad_cat(dy, w, Ca, out_dtype=L.DT_F32, path=L.PATH_TENSOR, za_in=za, zb_in=zb,
                             act_in=1)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)
    got = np.concatenate([host(gxa), host(gxb)], axis=-1)
    assert rel_err(got, ref) <= TOL_BF16


def test_pks_fused_concat_and_strided(monkeypatch):
    # the concat-free calls (a chunk pair across the split), the fused activation
    # backward and a stride-2 forward on K-split pair tiles
    monkeypatch.setenv("CONV3X3_PKS", "1")
    shape = (2, 192, 64, 256, 6, 7)  # N, Ca, Cb, Cout, H, W
    N, Ca, Cb, Cout, H, W = shape
    t, zin_h, _ = _cat_case(shape)
    x, w, b, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    y32 = ops.fwd_cat(xa, xb, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd_cat(t.x[..., :Ca], t.x[..., Ca:], t.w, t.bias, 1)) <= TOL_BF16
    zin = to_dev_bf16(zin_h)
    za, zb = zin[..., :Ca].contiguous(), zin[..., Ca:].contiguous()
    gxa, gxb = ops.dgrad_cat(dy, w, Ca, out_dtype=L.DT_F32, path=L.PATH_TENSOR, za_in=za, zb_in=zb,
                             act_in=1)
    torch.cuda.synchronize()
    got = np.concatenate([host(gxa), host(gxb)], axis=-1)
    assert rel_err(got, oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)) <= TOL_BF16
    ts = _small((2, 256, 256, 9, 9), seed=53)
    xs, ws, bs, _ = dev_tensors(ts)
    ys = ops.fwd_strided(xs, ws, bs, stride=2, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(ys), oracle.conv3x3_fwd_strided(ts.x, ts.w, ts.bias, 1, 2)) <= TOL_BF16


HALO_SHAPES = [
    (2, 64, 64, 16, 16),    # W = 16: one tile = one whole image
    (1, 72, 200, 8, 32),    # W = 32, ragged channel chunk and ragged N tile
    (2, 128, 128, 4, 64),   # W = 64, tiles of 4 rows
    (3, 8, 128, 16, 16),    # 8 input channels
    (1, 192, 256, 32, 32),  # several tiles per image, 3 channel chunks
]


@pytest.mark.parametrize("tile", ["halo64", "halo128"])
@pytest.mark.parametrize("shape", HALO_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_halo_tiles(shape, tile, monkeypatch):
    monkeypatch.setenv("CONV3X3_TILE", tile)
    t = _small(shape)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    ybf = ops.fwd(x, w, b, act=1, path=L.PATH_TENSOR)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)
    assert rel_err(host(y32), ref) <= TOL_BF16
    assert np.array_equal(host(ybf), rne_bf16(host(y32)))
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16
    yl = ops.fwd(x, w, b, act=L.ACT_LRELU, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(yl), oracle.conv3x3_fwd(t.x, t.w, t.bias, 2)) <= TOL_BF16


STEM_SHAPES = [
    (2, 8, 24, 9, 9),     # Cout 24 < 64: one mostly-empty N tile, ragged pixel tail
    (1, 8, 64, 7, 5),
    (2, 8, 256, 8, 8),    # the widest single N tile
    (3, 8, 128, 1, 13),   # single-row images
    (5, 8, 128, 16, 16),  # several 128-pixel tiles per CTA
    (2, 8, 72, 9, 11),    # 128-channel tile, second 64-channel store box clipped to 8 channels
    (1, 8, 104, 13, 10),  # clipped store box and a ragged pixel tail
    # widths 64 and 32 with whole-row tiles: the forward stages x as image rows
    (2, 8, 128, 4, 64),
    (1, 8, 72, 8, 32),
    (2, 8, 256, 2, 64),   # 256-channel tile
    (3, 8, 40, 4, 32),    # 64-channel tile
]


@pytest.mark.parametrize("rows", ["auto", "0"], ids=["rows_auto", "im2col"])
@pytest.mark.parametrize("shape", STEM_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_eight_channel_kernels(shape, rows, monkeypatch):
    if rows == "0":
        monkeypatch.setenv("CONV3X3_STEM_ROWS", "0")
    t = _small(shape)
    x, w, b, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert rel_err(host(dx32), oracle.conv3x3_dgrad(t.dy, t.w)) <= TOL_BF16
    for act in (0, 1, 2):
        y32 = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
        ybf = ops.fwd(x, w, b, act=act, path=L.PATH_TENSOR)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_fwd(t.x, t.w, t.bias, act)
        assert rel_err(host(y32), ref) <= TOL_BF16
        assert check_bf16_store(host(ybf), ref) == 0
        assert np.array_equal(host(ybf), rne_bf16(host(y32)))


STEM_WGRAD_SHAPES = [
    # width 64: each 64-pixel k-block is one image row
    (2, 8, 128, 4, 64),
    (2, 8, 256, 2, 64),   # two 128-channel tiles
    (1, 8, 24, 3, 64),    # Cout 24: a mostly empty tile
    (3, 8, 200, 5, 64),   # ragged second tile
    (2, 8, 128, 1, 64),   # single-row images: both halo rows are padding
]


@pytest.mark.parametrize("mode", ["halo", "im2col"])
@pytest.mark.parametrize("shape", STEM_WGRAD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_eight_channel_wgrad_x_layouts(shape, mode, monkeypatch):
    if mode == "im2col":
        monkeypatch.setenv("CONV3X3_STEM_ROWS", "0")
    t = _small(shape, seed=29)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    dw2, db2 = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.equal(dw, dw2) and torch.equal(db, db2)


# ---------------------------------------------------------------------------
# backward through the input's activation, fused into the epilogues
# ---------------------------------------------------------------------------
FUSED_SHAPES = [
    (2, 64, 64, 9, 9),
    (1, 72, 200, 6, 11),    # ragged channel chunks and N tiles
    (2, 8, 128, 12, 12),    # eight input channels: dgrad writes 8 channels
    (3, 128, 256, 17, 13),
    (2, 256, 64, 5, 7),
    (3, 8, 128, 5, 64),     # eight input channels, width 64: the row-band dgrad
]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fused_activation_backward(shape, path):
    p = PATHS[path]
    N, Cin, Cout, H, W = shape
    t = _small(shape)
    zin_h = synth.make_zin(t.layer, seed=7)
    x, w, b, dy = dev_tensors(t)
    zin = to_dev_bf16(zin_h)
    for act in (1, 2):
        # forward that also keeps z: y unchanged, z = the act-free output, bit for bit
        z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
        y = ops.fwd(x, w, b, act=act, path=p, z_out=z)
        y_plain = ops.fwd(x, w, b, act=act, path=p)
        z_plain = ops.fwd(x, w, b, act=0, path=p)
        torch.cuda.synchronize()
        assert torch.equal(y, y_plain), act
        assert torch.equal(z, z_plain), act
        assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) == 0
        # dgrad scaled by act'(z_in)
        dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p, z_in=zin, act_in=act)
        dxbf = ops.dgrad(dy, w, path=p, z_in=zin, act_in=act)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, act)
        assert rel_err(host(dx32), ref) <= TOL_BF16, act
        assert check_bf16_store(host(dxbf), ref) == 0, act
        assert np.array_equal(host(dxbf), rne_bf16(host(dx32))), act
    # act_in = NONE is plain dgrad (z_in ignored)
    dxn = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p, z_in=zin, act_in=L.ACT_NONE)
    dxp = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p)
    torch.cuda.synchronize()
    assert torch.equal(dxn, dxp)


@pytest.mark.parametrize("tile", ["64x2", "256x1", "256x1n", "halo64", "128x2", "128x2n", "pair128",
                                  "pair192", "pair384"])
def test_fused_activation_backward_tiles(tile, monkeypatch):
    monkeypatch.setenv("CONV3X3_TILE", tile)
    shape = (2, 64, 128, 16, 16)
    N, Cin, Cout, H, W = shape
    t = _small(shape)
    zin_h = synth.make_zin(t.layer, seed=7)
    x, w, b, dy = dev_tensors(t)
    z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
    y = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR, z_out=z)
    dx = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR, z_in=to_dev_bf16(zin_h),
                   act_in=1)
    torch.cuda.synchronize()
    assert rel_err(host(y), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) <= TOL_BF16
    assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) == 0
    assert rel_err(host(dx), oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)) <= TOL_BF16


# dgrad with 8 output channels and whole-row tiles of 128 pixels (the stem's
# input gradient): T = dy x Wt on the tensor cores, then the nine-tap sum
# CONV3X3_STEM_DGRAD=rows runs width 64 as row bands (T formed once per dy row,
# a ring of staged T rows; bands cross image boundaries); by default, tiles.
STEM_DGRAD_SHAPES = [
    (2, 8, 128, 64, 64),   # two dx rows per tile / bands of one row (128 rows, 128+ SMs)
    (3, 8, 64, 8, 32),     # 64 dy channels, four rows per tile
    (4, 8, 128, 16, 8),    # sixteen rows of width 8 per tile
    (2, 8, 128, 2, 64),    # one tile per image: both halo rows outside it
    (64, 8, 128, 7, 64),   # 448 rows: bands of three rows crossing image boundaries
    (5, 8, 64, 3, 64),     # 64 dy channels, odd image height, one-row bands
]


@pytest.mark.parametrize("kernel", ["tiles", "rows"])
@pytest.mark.parametrize("shape", STEM_DGRAD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_eight_output_channel_dgrad(shape, kernel, monkeypatch):
    if kernel == "rows":
        monkeypatch.setenv("CONV3X3_STEM_DGRAD", "rows")
    t = _small(shape)
    zin_h = synth.make_zin(t.layer, seed=7)
    x, w, b, dy = dev_tensors(t)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    dxbf = ops.dgrad(dy, w, path=L.PATH_TENSOR)
    ga = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=L.PATH_TENSOR, z_in=to_dev_bf16(zin_h), act_in=1)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_dgrad(t.dy, t.w)
    assert rel_err(host(dx32), ref) <= TOL_BF16
    assert check_bf16_store(host(dxbf), ref) == 0
    assert np.array_equal(host(dxbf), rne_bf16(host(dx32)))
    assert rel_err(host(ga), oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)) <= TOL_BF16


@pytest.mark.parametrize("path", sorted(PATHS))
def test_wgrad_is_bit_deterministic(path):
    t = _small((4, 128, 128, 16, 16))
    x, _, _, dy = dev_tensors(t)
    a = ops.wgrad(x, dy, path=PATHS[path])
    b = ops.wgrad(x, dy, path=PATHS[path])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# The weight gradient's two x layouts: im2col boxes per tap, and (stride 1,
# width 16, 32 or 64) one zero-padded box of W + 2 columns per image row that
# all three taps of a kernel row read, shifted by a row each.
WGRAD_ROW_SHAPES = [
    (1, 128, 128, 4, 16),   # 16-wide rows, four per k-block
    (2, 64, 128, 2, 32),    # 32-wide rows, two per k-block
    (1, 128, 64, 1, 64),    # one 64-wide row: kernel rows 0 and 2 read only padding
    (2, 256, 256, 4, 16),   # several channel blocks and tiles
    (1, 72, 200, 8, 16),    # ragged channel box and ragged Cout block
    (3, 64, 64, 6, 32),     # several splits over several images
]


@pytest.mark.parametrize("rows", ["1", "0"], ids=["row_shifted", "im2col"])
@pytest.mark.parametrize("shape", WGRAD_ROW_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_wgrad_x_layouts(shape, rows, monkeypatch):
    monkeypatch.setenv("CONV3X3_WGRAD_ROWS", rows)
    t = _small(shape, seed=13)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    dw2, db2 = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.equal(dw, dw2) and torch.equal(db, db2)


WGRAD_PAIR_SHAPES = [
    # N, Cin, Cout, H, W: Cout a multiple of 256 takes the two-CTA tiles
    (2, 128, 256, 8, 8),     # one pair block
    (1, 64, 512, 5, 7),      # ragged pixel tail, half a channel block, two pair blocks
    (2, 192, 256, 6, 10),    # ragged channel block (128 + 64)
    (1, 72, 256, 9, 9),      # ragged 64-channel box
    (3, 256, 256, 16, 16),   # several channel blocks and splits
]


@pytest.mark.parametrize("pair", ["1", "0"], ids=["pair", "one_cta"])
@pytest.mark.parametrize("shape", WGRAD_PAIR_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_wgrad_pair_tiles(shape, pair, monkeypatch):
    monkeypatch.setenv("CONV3X3_WGRAD_PAIR", pair)
    t = _small(shape, seed=19)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    dw2, db2 = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.equal(dw, dw2) and torch.equal(db, db2)


WGRAD_HYBRID_SHAPES = [
    # N, Cin, Cout, H, W: Cout above 256 and not a multiple of it -- pair tiles
    # over the first 256 k output channels, one-CTA tiles over the rest
    (2, 128, 384, 8, 8),     # 256 + one 128-channel block
    (1, 64, 320, 5, 7),      # 256 + half a block, ragged pixel tail
    (1, 72, 448, 9, 9),      # 256 + one and a half blocks, ragged 64-channel box
    (3, 256, 384, 16, 16),   # several channel blocks and splits
    (1, 192, 640, 6, 6),     # 512 + 128: two pair blocks
]


@pytest.mark.parametrize("hybrid", ["1", "0"], ids=["hybrid", "one_cta"])
@pytest.mark.parametrize("shape", WGRAD_HYBRID_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_wgrad_hybrid_tiles(shape, hybrid, monkeypatch):
    # the two parts have split plans of their own; dw rows and dbias entries
    # of each part are summed over that part's splits only
    monkeypatch.setenv("CONV3X3_WGRAD_HYBRID", hybrid)
    t = _small(shape, seed=29)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    dw2, db2 = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.equal(dw, dw2) and torch.equal(db, db2)


@pytest.mark.parametrize("splits", ["1", "5"])
def test_wgrad_hybrid_forced_splits_and_concat(splits, monkeypatch):
    # one split count forced on both parts, and x from two tensors
    monkeypatch.setenv("CONV3X3_WGRAD_SPLITS", splits)
    N, Ca, Cb, Cout, H, W = 1, 128, 64, 384, 8, 10
    t = _small((N, Ca + Cb, Cout, H, W), seed=31)
    x, _, _, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    dw, db = ops.wgrad_cat(xa, xb, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16


@pytest.mark.parametrize("splits", ["1", "3", "10"])
def test_wgrad_pair_split_counts(splits, monkeypatch):
    # 624 pixels = 10 k-blocks, the last one 48 pixels: one split, splits of
    # 4 + 4 + 2 k-blocks, one k-block per split
    monkeypatch.setenv("CONV3X3_WGRAD_SPLITS", splits)
    t = _small((3, 128, 256, 13, 16), seed=23)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16


@pytest.mark.parametrize("path", sorted(PATHS))
def test_wgrad_dbias_only_four_byte_aligned(path):
    # dbias may sit 4 bytes past a 16-byte boundary (the ABI asks for 4)
    t = _small((2, 64, 136, 8, 8), seed=17)
    x, _, _, dy = dev_tensors(t)
    dw = torch.empty((136, 3, 3, 64), dtype=torch.float32, device="cuda")
    buf = torch.full((137 + 3,), float("nan"), dtype=torch.float32, device="cuda")
    db = buf[1:137]
    assert db.data_ptr() % 16 == 4
    ops.wgrad(x, dy, path=PATHS[path], out=(dw, db))
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.isnan(buf[0]) and torch.all(torch.isnan(buf[137:]))  # nothing written outside


def test_wgrad_without_dbias_and_dirty_workspace():
    t = _small((2, 64, 128, 8, 8))
    x, _, _, dy = dev_tensors(t)
    ws = ops.wgrad_workspace(2, 64, 128, 8, 8)
    ws[0].fill_(0x7F)  # garbage in the scratch must not matter
    dw, db = ops.wgrad(x, dy, with_bias=False, workspace=ws)
    torch.cuda.synchronize()
    assert db is None
    assert rel_err(host(dw), oracle.conv3x3_wgrad(t.x, t.dy)[0]) <= TOL_BF16


def test_stem_padded_channels_stay_zero():
    Lr = synth.Layer("stem-mini", 4, 8, 128, 16, 16, act=1, cin_real=3)
    t = synth.make_tensors(Lr, seed=3)
    x, w, b, dy = dev_tensors(t)
    for p in PATHS.values():
        dx = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p)
        dw, _ = ops.wgrad(x, dy, path=p)
        torch.cuda.synchronize()
        assert torch.all(dx[..., 3:] == 0)
        assert torch.all(dw[..., 3:] == 0)


def test_bad_channel_count_is_rejected():
    x = torch.zeros((1, 4, 4, 12), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 3, 3, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.Conv3x3Error) as e:
        ops.fwd(x, w)
    assert e.value.status == L.ERR_INVALID_ARG


def test_bounded_wait_times_out_and_context_survives():
    assert L.conv3x3_device_status() == L.OK
    L.conv3x3_selftest_wait_timeout(2_000_000)  # 2 ms, on a barrier nobody arrives at
    assert L.conv3x3_device_status() == L.ERR_TIMEOUT
    assert L.conv3x3_device_status() == L.OK  # read-and-clear
    t = _small((1, 64, 64, 4, 4))
    x, w, b, _ = dev_tensors(t)
    y = ops.fwd(x, w, b, act=0, out_dtype=L.DT_F32)
    torch.cuda.synchronize()
    assert rel_err(host(y), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) <= TOL_BF16


# ---------------------------------------------------------------------------
# full-size workloads, sampled outputs, AUTO path (what the benchmark runs)
# ---------------------------------------------------------------------------
def _sampled_layer_check(Lr, seed, index, n_rand=4096, dw_rows=None, whole_images=True):
    """y and dx: n_rand random outputs (+ every output of the first and last
    image, which hold every border and corner); dw and db: every element
    (dw_rows None) or the full [3][3][Cin] rows of the output channels in
    dw_rows -- the oracle's wgrad of dy restricted to those channels, since
    dw[k] depends on dy[..., k] alone."""
    t = synth.make_tensors(Lr, seed=seed, index=index)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd(x, w, b, act=Lr.act, out_dtype=L.DT_F32)
    ybf = ops.fwd(x, w, b, act=Lr.act)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32)
    dw, db = ops.wgrad(x, dy)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1000 + index)
    y32h, ybfh, dxh = host(y32).reshape(-1), host(ybf).reshape(-1), host(dx32).reshape(-1)
    per_img_y = Lr.H * Lr.W * Lr.Cout
    per_img_x = Lr.H * Lr.W * Lr.Cin
    iy = rng.integers(0, y32h.size, n_rand)
    ix = rng.integers(0, dxh.size, n_rand)
    if whole_images:
        iy = np.concatenate([iy, np.arange(per_img_y), np.arange(y32h.size - per_img_y, y32h.size)])
        ix = np.concatenate([ix, np.arange(per_img_x), np.arange(dxh.size - per_img_x, dxh.size)])
    ry = oracle.conv3x3_fwd_at(t.x, t.w, t.bias, Lr.act, iy)
    scale_y = max(np.max(np.abs(ry)), 1e-30)
    assert np.max(np.abs(y32h[iy] - ry)) / scale_y <= TOL_BF16, Lr.name
    assert np.array_equal(ybfh[iy], rne_bf16(y32h[iy])), Lr.name
    rx = oracle.conv3x3_dgrad_at(t.dy, t.w, ix)
    assert np.max(np.abs(dxh[ix] - rx)) / max(np.max(np.abs(rx)), 1e-30) <= TOL_BF16, Lr.name
    dwh, dbh = host(dw), host(db)
    if dw_rows is None:
        rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
        assert rel_err(dwh, rdw) <= TOL_BF16, Lr.name
        assert rel_err(dbh, rdb) <= TOL_BF16, Lr.name
    else:
        ks = np.asarray(sorted(set(dw_rows)))
        rdw, rdb = oracle.conv3x3_wgrad(t.x, np.ascontiguousarray(t.dy[..., ks]))
        assert rel_err(dwh[ks], rdw) <= TOL_BF16, Lr.name
        assert rel_err(dbh, oracle.conv3x3_dbias(t.dy)) <= TOL_BF16, Lr.name


@pytest.mark.parametrize("name", ["stem", "l1", "l2", "l3"])
def test_full_size_configs_sampled(name):
    # y and dx sampled (two whole images + random outputs), all of dw and db
    Lr = synth.CONFIGS[name][0]
    _sampled_layer_check(Lr, seed=0, index=0)


def test_fused_activation_backward_full_size_sampled():
    # the 128-channel 64x64 layer at batch 64, AUTO path, as the fused step runs it
    Lr = synth.L1
    t = synth.make_tensors(Lr, seed=0, index=0)
    zin_h = synth.make_zin(Lr, seed=0, index=0)
    x, w, b, dy = dev_tensors(t)
    z = torch.empty((Lr.N, Lr.H, Lr.W, Lr.Cout), dtype=torch.bfloat16, device="cuda")
    ops.fwd(x, w, b, act=1, z_out=z)
    dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, z_in=to_dev_bf16(zin_h), act_in=1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(77)
    zh, dxh = host(z).reshape(-1), host(dx32).reshape(-1)
    iz = rng.integers(0, zh.size, 4096)
    rz = oracle.conv3x3_fwd_at(t.x, t.w, t.bias, 0, iz)
    assert check_bf16_store(zh[iz], rz) == 0
    ix = rng.integers(0, dxh.size, 4096)
    rx = oracle.conv3x3_dgrad_act_at(t.dy, t.w, zin_h, 1, ix)
    assert np.max(np.abs(dxh[ix] - rx)) / max(np.max(np.abs(rx)), 1e-30) <= TOL_BF16


# ---------------------------------------------------------------------------
# the epilogue's activations far from zero: SiLU and leaky ReLU forwards and the
# fused activation backward with pre-activations near +-30, +-90 and +-200,
# where exp(-z) overflows or underflows in fp32
# ---------------------------------------------------------------------------
SAT_LEVELS = np.array([-200.0, -90.0, -30.0, -3.0, 3.0, 30.0, 90.0, 200.0])
SAT_CASES = [
    # (id, (N, Cin, Cout, H, W), forced tile or None)
    ("default", (2, 64, 64, 8, 8), None),
    ("transposed", (2, 64, 128, 16, 16), "128x2"),
    ("pair", (2, 64, 256, 16, 16), "256x1"),
    ("stem", (2, 8, 128, 16, 16), None),
]


def _grouped_ok(got, ref, groups):
    """Every value finite, and per channel group (channels with one level)
    max|err| <= 2e-3 * max(max|ref| of the group, 1e-3 * max|ref| overall):
    each saturated group is held to its own scale, not to the largest one."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not np.all(np.isfinite(got)):
        return False
    C = ref.shape[-1]
    g2, r2 = got.reshape(-1, C), ref.reshape(-1, C)
    floor = 1e-3 * np.max(np.abs(r2))
    for g in range(groups):
        cols = np.arange(g, C, groups)
        scale = max(np.max(np.abs(r2[:, cols])), floor)
        if np.max(np.abs(g2[:, cols] - r2[:, cols])) > TOL_BF16 * scale:
            return False
    return True


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("case", SAT_CASES, ids=lambda c: c[0])
def test_activations_in_their_saturated_range(case, path, monkeypatch):
    _, shape, tile = case
    p = PATHS[path]
    if tile is not None:
        if p == L.PATH_SIMT:
            pytest.skip("the tile override only concerns the tensor-core kernels")
        monkeypatch.setenv("CONV3X3_TILE", tile)
    N, Cin, Cout, H, W = shape
    t = _small(shape, seed=21)
    ng = len(SAT_LEVELS)
    # bias puts output channel k near SAT_LEVELS[k % 8]; z_in puts input channel
    # c near SAT_LEVELS[c % 8] (rounded to bf16 like every activation)
    bias = (SAT_LEVELS[np.arange(Cout) % ng] + t.bias).astype(np.float32)
    zin = synth.bf16_round((SAT_LEVELS[np.arange(Cin) % ng]
                            + np.random.default_rng(5).standard_normal((N, H, W, Cin))).astype(np.float32))
    x, w, _, dy = dev_tensors(t)
    b = to_dev_f32(bias)
    for act in (1, 2):
        z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
        y32 = ops.fwd(x, w, b, act=act, out_dtype=L.DT_F32, path=p, z_out=z)
        ybf = ops.fwd(x, w, b, act=act, path=p)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_fwd(t.x, t.w, bias, act)
        assert _grouped_ok(host(y32), ref, ng), ("fwd", act)
        assert check_bf16_store(host(ybf), ref) == 0, ("fwd bf16 store", act)
        assert np.array_equal(host(ybf), rne_bf16(host(y32))), ("fwd one rounding", act)
        assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, bias, 0)) == 0, ("z", act)
        dx32 = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p, z_in=to_dev_bf16(zin), act_in=act)
        torch.cuda.synchronize()
        rdx = oracle.conv3x3_dgrad_act(t.dy, t.w, zin, act)
        assert _grouped_ok(host(dx32), rdx, ng), ("dgrad_act", act)


def test_full_unet_stack_sampled():
    # every layer of the benchmark step: the first and last image of y and dx,
    # random outputs, and full dw rows of the first, a middle and the last
    # output channel (a split-range or tail-tile slip in wgrad shows in every row)
    for i, Lr in enumerate(synth.UNET_STEP):
        _sampled_layer_check(Lr, seed=0, index=i, n_rand=1024,
                             dw_rows=(0, Lr.Cout // 2 + 1, Lr.Cout - 1), whole_images=True)


# ---------------------------------------------------------------------------
# channel-concatenated input passed as two tensors (UNet up-path convs)
# ---------------------------------------------------------------------------
CAT_SHAPES = [
    # N, Ca, Cb, Cout, H, W
    (2, 64, 64, 64, 9, 9),
    (1, 128, 72, 200, 6, 11),   # ragged second part and N tiles
    (2, 256, 128, 128, 8, 8),
    (1, 64, 192, 96, 5, 7),
    (2, 24, 40, 64, 6, 6),      # Ca not a whole 64-channel chunk: CUDA-core kernels only
    (1, 64, 128, 128, 4, 16),   # wgrad with row-shifted x boxes from both parts
    (2, 128, 64, 64, 2, 32),
    (2, 128, 64, 256, 6, 6),    # wgrad on two-CTA tiles, x from both parts
]


def _cat_case(shape, seed=11):
    N, Ca, Cb, Cout, H, W = shape
    t = _small((N, Ca + Cb, Cout, H, W), seed=seed)
    zin = synth.make_zin(t.layer, seed=seed)
    return t, zin, Ca


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", CAT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_concat_free_convs(shape, path):
    p = PATHS[path]
    N, Ca, Cb, Cout, H, W = shape
    Cin = Ca + Cb
    t, zin_h, _ = _cat_case(shape)
    x, w, b, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    if p == L.PATH_TENSOR and Ca % 64:
        with pytest.raises(L.Conv3x3Error) as e:
            ops.fwd_cat(xa, xb, w, b, act=1, path=p)
        assert e.value.status == L.ERR_UNSUPPORTED
        return
    # forward: equals the oracle on the concatenation, and the plain kernel on
    # the materialised concatenation bit for bit (same tiles, same K order)
    z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
    y32 = ops.fwd_cat(xa, xb, w, b, act=1, out_dtype=L.DT_F32, path=p, z_out=z)
    y32_plain = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32, path=p)
    z_plain = ops.fwd(x, w, b, act=0, path=p)
    torch.cuda.synchronize()
    ta, tb = t.x[..., :Ca], t.x[..., Ca:]
    assert rel_err(host(y32), oracle.conv3x3_fwd_cat(ta, tb, t.w, t.bias, 1)) <= TOL_BF16
    assert torch.equal(y32, y32_plain)
    assert torch.equal(z, z_plain)
    # input gradient, split; plain and through the activation
    dxa, dxb = ops.dgrad_cat(dy, w, Ca, out_dtype=L.DT_F32, path=p)
    dx_plain = ops.dgrad(dy, w, out_dtype=L.DT_F32, path=p)
    torch.cuda.synchronize()
    ra, rb = oracle.conv3x3_dgrad_cat(t.dy, t.w, Ca)
    scale = max(np.max(np.abs(ra)), np.max(np.abs(rb)))
    assert np.max(np.abs(host(dxa) - ra)) / scale <= TOL_BF16
    assert np.max(np.abs(host(dxb) - rb)) / scale <= TOL_BF16
    assert torch.equal(dxa, dx_plain[..., :Ca]) and torch.equal(dxb, dx_plain[..., Ca:])
    zin = to_dev_bf16(zin_h)
    za, zb = zin[..., :Ca].contiguous(), zin[..., Ca:].contiguous()
    gxa, gxb = ops.dgrad_cat(dy, w, Ca, path=p, za_in=za, zb_in=zb, act_in=1)
    gx_plain = ops.dgrad(dy, w, path=p, z_in=zin, act_in=1)
    torch.cuda.synchronize()
    assert torch.equal(gxa, gx_plain[..., :Ca]) and torch.equal(gxb, gx_plain[..., Ca:])
    ref = oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)
    assert check_bf16_store(np.concatenate([host(gxa), host(gxb)], axis=-1), ref) == 0
    # weight gradient: oracle, and bit-identical to the plain call on the concatenation
    dw, db = ops.wgrad_cat(xa, xb, dy, path=p)
    dw_plain, db_plain = ops.wgrad(x, dy, path=p)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad_cat(ta, tb, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
    assert torch.equal(dw, dw_plain) and torch.equal(db, db_plain)


@pytest.mark.parametrize("tile", ["128x2", "128x2n", "256x1", "256x1n", "pair192", "pair384"])
@pytest.mark.parametrize("shape", [(1, 128, 72, 200, 6, 11), (2, 128, 128, 128, 16, 16),
                                   (1, 192, 64, 256, 6, 7)],  # a two-chunk stage across the split
                         ids=lambda s: "x".join(map(str, s)))
def test_concat_free_256_pixel_tiles(shape, tile, monkeypatch):
    """Split input and split input gradient on the 256-pixel tiles: transposed
    (one channel per epilogue thread) and not, on CTA pairs and on one CTA."""
    monkeypatch.setenv("CONV3X3_TILE", tile)
    N, Ca, Cb, Cout, H, W = shape
    t, zin_h, _ = _cat_case(shape)
    x, w, b, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    y32 = ops.fwd_cat(xa, xb, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd_cat(t.x[..., :Ca], t.x[..., Ca:], t.w, t.bias, 1)) <= TOL_BF16
    zin = to_dev_bf16(zin_h)
    za, zb = zin[..., :Ca].contiguous(), zin[..., Ca:].contiguous()
    gxa, gxb = ops.dgrad_cat(dy, w, Ca, out_dtype=L.DT_F32, path=L.PATH_TENSOR, za_in=za, zb_in=zb,
                             act_in=1)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_dgrad_act(t.dy, t.w, zin_h, 1)
    got = np.concatenate([host(gxa), host(gxb)], axis=-1)
    assert rel_err(got, ref) <= TOL_BF16


def test_concat_free_up_path_layer_full_size_sampled():
    # up1.rb0.conv1 of the UNet: main 384 + skip 256 channels at 32x32, batch 64
    i, Lr = next((i, Lr) for i, Lr in enumerate(synth.UNET_STEP) if Lr.name == "up1.rb0.conv1")
    Ca = Lr.cat_a
    assert Ca == 384
    t = synth.make_tensors(Lr, seed=0, index=i)
    x, w, b, dy = dev_tensors(t)
    xa, xb = x[..., :Ca].contiguous(), x[..., Ca:].contiguous()
    del x
    y32 = ops.fwd_cat(xa, xb, w, b, act=Lr.act, out_dtype=L.DT_F32)
    dxa, dxb = ops.dgrad_cat(dy, w, Ca, out_dtype=L.DT_F32)
    dw, db = ops.wgrad_cat(xa, xb, dy)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    ta, tb = t.x[..., :Ca], t.x[..., Ca:]
    yh = host(y32).reshape(-1)
    iy = rng.integers(0, yh.size, 2048)
    ry = oracle.conv3x3_fwd_cat_at(ta, tb, t.w, t.bias, Lr.act, iy)
    assert np.max(np.abs(yh[iy] - ry)) / np.max(np.abs(ry)) <= TOL_BF16
    dxh = np.concatenate([host(dxa), host(dxb)], axis=-1).reshape(-1)
    ix = rng.integers(0, dxh.size, 2048)
    rx = oracle.conv3x3_dgrad_at(t.dy, t.w, ix)
    assert np.max(np.abs(dxh[ix] - rx)) / np.max(np.abs(rx)) <= TOL_BF16
    dwh = host(dw).reshape(-1)
    iw = rng.integers(0, dwh.size, 64)
    rw = oracle.conv3x3_wgrad_cat_at(ta, tb, t.dy, iw)
    assert np.max(np.abs(dwh[iw] - rw)) / np.max(np.abs(rw)) <= TOL_BF16
    assert rel_err(host(db), oracle.conv3x3_dbias(t.dy)) <= TOL_BF16


# ---------------------------------------------------------------------------
# strided (downsampling) convolution
# ---------------------------------------------------------------------------
STRIDE_SHAPES = [
    # N, Cin, Cout, H, W
    (2, 64, 64, 8, 8),
    (1, 72, 200, 7, 9),     # odd grid, ragged channel chunk and N tiles
    (2, 128, 128, 16, 16),
    (3, 64, 96, 5, 6),
    (1, 64, 64, 1, 5),      # single-row images
    (2, 16, 32, 6, 7),      # fewer than 64 channels: CUDA-core kernels only
    (2, 64, 256, 9, 9),     # wgrad on two-CTA tiles
]


def _strided_case(shape, seed=13):
    N, Cin, Cout, H, W = shape
    Lr = synth.Layer("s2", N, Cin, Cout, H, W, act=1, stride=2)
    return synth.make_tensors(Lr, seed=seed), synth.make_zin(Lr, seed=seed)


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", STRIDE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stride_two_convs(shape, path):
    p = PATHS[path]
    N, Cin, Cout, H, W = shape
    Ho, Wo = (H + 1) // 2, (W + 1) // 2
    t, zin_h = _strided_case(shape)
    x, w, b, dy = dev_tensors(t)
    assert tuple(dy.shape) == (N, Ho, Wo, Cout)
    if p == L.PATH_TENSOR and min(Cin, Cout) < 64:
        with pytest.raises(L.Conv3x3Error) as e:
            ops.fwd_strided(x, w, b, act=1, path=p)
        assert e.value.status == L.ERR_UNSUPPORTED
        return
    for act in (0, 1):
        z = torch.empty((N, Ho, Wo, Cout), dtype=torch.bfloat16, device="cuda")
        y32 = ops.fwd_strided(x, w, b, act=act, out_dtype=L.DT_F32, path=p)
        ybf = ops.fwd_strided(x, w, b, act=act, path=p, z_out=z)
        torch.cuda.synchronize()
        ref = oracle.conv3x3_fwd_strided(t.x, t.w, t.bias, act, u=2)
        assert rel_err(host(y32), ref) <= TOL_BF16, act
        assert check_bf16_store(host(ybf), ref) == 0, act
        assert np.array_equal(host(ybf), rne_bf16(host(y32))), act
        assert check_bf16_store(host(z), oracle.conv3x3_fwd_strided(t.x, t.w, t.bias, 0, u=2)) == 0
    dx32 = ops.dgrad_strided(dy, w, H, W, out_dtype=L.DT_F32, path=p)
    dxbf = ops.dgrad_strided(dy, w, H, W, path=p)
    torch.cuda.synchronize()
    ref = oracle.conv3x3_dgrad_strided(t.dy, t.w, H, W, u=2)
    assert rel_err(host(dx32), ref) <= TOL_BF16
    assert check_bf16_store(host(dxbf), ref) == 0
    assert np.array_equal(host(dxbf), rne_bf16(host(dx32)))
    ga = ops.dgrad_strided(dy, w, H, W, out_dtype=L.DT_F32, path=p, z_in=to_dev_bf16(zin_h),
                           act_in=1)
    torch.cuda.synchronize()
    grad = oracle.act_grad
    ref_a = ref * np.vectorize(lambda z: grad(1, z))(zin_h.astype(np.float64))
    assert rel_err(host(ga), ref_a) <= TOL_BF16
    dw, db = ops.wgrad_strided(x, dy, path=p)
    torch.cuda.synchronize()
    rdw, rdb = oracle.conv3x3_wgrad_strided(t.x, t.dy, u=2)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16


@pytest.mark.parametrize("path", sorted(PATHS))
def test_stride_one_through_the_strided_calls_is_the_plain_call(path):
    p = PATHS[path]
    t = _small((2, 64, 64, 9, 7))
    x, w, b, dy = dev_tensors(t)
    assert torch.equal(ops.fwd_strided(x, w, b, stride=1, act=1, path=p), ops.fwd(x, w, b, act=1, path=p))
    assert torch.equal(ops.dgrad_strided(dy, w, 9, 7, stride=1, path=p), ops.dgrad(dy, w, path=p))
    dw1, db1 = ops.wgrad_strided(x, dy, stride=1, path=p)
    dw0, db0 = ops.wgrad(x, dy, path=p)
    assert torch.equal(dw1, dw0) and torch.equal(db1, db0)


@pytest.mark.parametrize("tile", ["64x1", "128x2", "256x1", "256x1n"])
def test_stride_two_tiles(tile, monkeypatch):
    monkeypatch.setenv("CONV3X3_TILE", tile)
    shape = (2, 64, 128, 13, 10)
    N, Cin, Cout, H, W = shape
    t, _ = _strided_case(shape)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd_strided(x, w, b, act=1, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    dx32 = ops.dgrad_strided(dy, w, H, W, out_dtype=L.DT_F32, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd_strided(t.x, t.w, t.bias, 1, u=2)) <= TOL_BF16
    assert rel_err(host(dx32), oracle.conv3x3_dgrad_strided(t.dy, t.w, H, W, u=2)) <= TOL_BF16


@pytest.mark.parametrize("index", [0, 2])
def test_downsampling_layers_full_size_sampled(index):
    Lr = synth.DOWNSAMPLE[index]
    t = synth.make_tensors(Lr, seed=0, index=index)
    x, w, b, dy = dev_tensors(t)
    y32 = ops.fwd_strided(x, w, b, act=Lr.act, out_dtype=L.DT_F32)
    dx32 = ops.dgrad_strided(dy, w, Lr.H, Lr.W, out_dtype=L.DT_F32)
    dw, db = ops.wgrad_strided(x, dy)
    torch.cuda.synchronize()
    rng = np.random.default_rng(21 + index)
    yh, dxh, dwh = host(y32).reshape(-1), host(dx32).reshape(-1), host(dw).reshape(-1)
    iy = rng.integers(0, yh.size, 2048)
    ry = oracle.conv3x3_fwd_strided_at(t.x, t.w, t.bias, Lr.act, 2, iy)
    assert np.max(np.abs(yh[iy] - ry)) / np.max(np.abs(ry)) <= TOL_BF16
    per_img = Lr.H * Lr.W * Lr.Cin   # every dx of the first image (all four parity classes, borders)
    ix = np.concatenate([rng.integers(0, dxh.size, 2048), np.arange(min(per_img, 65536))])
    rx = oracle.conv3x3_dgrad_strided_at(t.dy, t.w, Lr.H, Lr.W, 2, ix)
    assert np.max(np.abs(dxh[ix] - rx)) / np.max(np.abs(rx)) <= TOL_BF16
    iw = rng.integers(0, dwh.size, 64)
    rw = oracle.conv3x3_wgrad_strided_at(t.x, t.dy, 2, iw)
    assert np.max(np.abs(dwh[iw] - rw)) / np.max(np.abs(rw)) <= TOL_BF16
    rdb = oracle.conv3x3_wgrad_strided_at(t.x, t.dy, 2, dwh.size + np.arange(Lr.Cout))
    assert rel_err(host(db), rdb) <= TOL_BF16


# Store paths.  The output and the weight gradient's split partials leave
# through TMA tensor stores where the library takes them; the per-thread store
# path that replaces them (CONV3X3_EPI_TMA=0, CONV3X3_WGRAD_PART_TMA=0) holds
# the same values, so both must give bit-identical tensors.
EPI_STORE_SHAPES = [
    # N, Cin, Cout, H, W: one tile per CTA (or CTA pair) for every tile kind
    (2, 64, 128, 12, 12),     # 128x1 tiles, ragged pixel tail
    (1, 256, 256, 16, 16),    # two-CTA 256-channel tiles
    (2, 384, 384, 16, 16),    # two-CTA 384-channel tiles
    (1, 128, 200, 9, 7),      # channels past the last 64-wide box are clipped
    (2, 512, 512, 8, 8),      # the 8x8 layer's tiles
]


@pytest.mark.parametrize("shape", EPI_STORE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_output_tma_stores_match_thread_stores(shape, monkeypatch):
    t = _small(shape, seed=37)
    x, w, b, dy = dev_tensors(t)
    zin = to_dev_bf16(synth.make_zin(t.layer, seed=37))  # laid out like dx

    def run():
        y = ops.fwd(x, w, b, act=1)
        dx = ops.dgrad(dy, w)
        gx = ops.dgrad(dy, w, z_in=zin, act_in=1)
        torch.cuda.synchronize()
        return y, dx, gx

    a = run()
    monkeypatch.setenv("CONV3X3_EPI_TMA", "0")
    c = run()
    for u, v in zip(a, c):
        assert torch.equal(u, v)
    y32 = ops.fwd(x, w, b, act=1, out_dtype=L.DT_F32)
    torch.cuda.synchronize()
    assert rel_err(host(y32), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) <= TOL_BF16


# Launches with more tiles than CTAs (or CTA pairs): each CTA's last tile
# leaves through TMA stores, the others through per-thread stores.  Forced
# tile kinds, ragged pixel tails and a ragged channel edge.
MULTI_TILE_STORE_CASES = [
    ("pair256", (10, 256, 256, 45, 45)),   # 80 two-CTA tiles over 76 pairs
    ("pair384", (80, 384, 384, 16, 16)),   # 80 two-CTA 384-channel tiles
    ("256x1n", (12, 256, 256, 45, 45)),    # 190 one-CTA 128 x 256 tiles
    ("128x1", (12, 128, 200, 45, 45)),     # 380 tiles, 200 channels (clipped box)
    ("128x2n", (20, 128, 128, 45, 45)),    # 159 untransposed 256 x 128 tiles
    ("64x2", (20, 64, 64, 45, 45)),        # 159 256 x 64 tiles
]


@pytest.mark.parametrize("tile,shape", MULTI_TILE_STORE_CASES, ids=lambda v: v if isinstance(v, str) else "x".join(map(str, v)))
def test_last_tile_tma_stores_match_thread_stores(tile, shape, monkeypatch):
    t = _small(shape, seed=41)
    x, w, b, dy = dev_tensors(t)
    zin = to_dev_bf16(synth.make_zin(t.layer, seed=41))
    monkeypatch.setenv("CONV3X3_TILE", tile)

    def run():
        y = ops.fwd(x, w, b, act=1)
        dx = ops.dgrad(dy, w)
        gx = ops.dgrad(dy, w, z_in=zin, act_in=1)
        torch.cuda.synchronize()
        return y, dx, gx

    a = run()
    monkeypatch.setenv("CONV3X3_EPI_TMA", "1")  # one-tile launches only: none here
    c = run()
    monkeypatch.setenv("CONV3X3_EPI_TMA", "0")
    e = run()
    for u, v, z in zip(a, c, e):
        assert torch.equal(u, v)
        assert torch.equal(u, z)
    # every channel of a few pixels in the last tiles against the oracle
    P, C = t.layer.N * t.layer.H * t.layer.W, t.layer.Cout
    pix = np.array([0, P - 257, P - 130, P - 2, P - 1])
    idx = (pix[:, None] * C + np.arange(C)[None, :]).reshape(-1)
    ry = oracle.conv3x3_fwd_at(t.x, t.w, t.bias, 1, idx)
    assert check_bf16_store(host(a[0]).reshape(-1)[idx], ry) == 0


STEM_Z_SHAPES = [
    (2, 8, 128, 8, 64),    # width 64: 128-pixel tiles of two image rows
    (3, 8, 128, 4, 32),    # width 32: four rows per tile
    (2, 8, 72, 8, 64),     # channels past the last 64-wide box are clipped
]


@pytest.mark.parametrize("shape", STEM_Z_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stem_forward_z_through_tma_stores(shape, monkeypatch):
    # the 8-input-channel forward storing z (the fused training step): y and z
    # through TMA tensor stores, against per-thread stores and the oracle
    t = _small(shape, seed=59)
    x, w, b, _ = dev_tensors(t)
    N, Cin, Cout, H, W = shape

    def run():
        z = torch.empty((N, H, W, Cout), dtype=torch.bfloat16, device="cuda")
        y = ops.fwd(x, w, b, act=1, path=L.PATH_TENSOR, z_out=z)
        torch.cuda.synchronize()
        return y, z

    y, z = run()
    monkeypatch.setenv("CONV3X3_STEM_ZTMA", "0")
    y0, z0 = run()
    assert torch.equal(y, y0) and torch.equal(z, z0)
    assert check_bf16_store(host(z), oracle.conv3x3_fwd(t.x, t.w, t.bias, 0)) == 0
    assert check_bf16_store(host(y), oracle.conv3x3_fwd(t.x, t.w, t.bias, 1)) == 0


WGRAD_STORE_SHAPES = [
    (2, 128, 128, 16, 16),    # one-CTA tiles, im2col x
    (2, 128, 128, 8, 64),     # one-CTA tiles, row-shifted x (width 64)
    (2, 128, 256, 8, 8),      # two-CTA tiles
    (1, 72, 200, 9, 9),       # ragged channel boxes (clipped columns and rows)
    (2, 128, 384, 8, 8),      # hybrid: two-CTA and one-CTA parts
    (2, 8, 128, 3, 64),       # 8 input channels, width 64: the stem kernel
    (1, 8, 136, 2, 64),       # the stem kernel with rows past Cout clipped
]


@pytest.mark.parametrize("shape", WGRAD_STORE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_wgrad_tma_partials_match_thread_stores(shape, monkeypatch):
    monkeypatch.setenv("CONV3X3_WGRAD_HYBRID", "1")
    t = _small(shape, seed=41)
    x, _, _, dy = dev_tensors(t)
    dw, db = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    monkeypatch.setenv("CONV3X3_WGRAD_PART_TMA", "0")
    dw2, db2 = ops.wgrad(x, dy, path=L.PATH_TENSOR)
    torch.cuda.synchronize()
    assert torch.equal(dw, dw2) and torch.equal(db, db2)
    rdw, rdb = oracle.conv3x3_wgrad(t.x, t.dy)
    assert rel_err(host(dw), rdw) <= TOL_BF16
    assert rel_err(host(db), rdb) <= TOL_BF16
