"""CPU oracle for the stride-1, pad-1 3x3 convolution (fwd, dgrad, dgrad through the
input's activation, wgrad, dbias).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the product path.

The arithmetic lives in ``conv3x3_oracle.c`` (plain fp64 loop nests, pthreads over
the outermost independent loop).  This module only compiles it with the host C
compiler and marshals numpy arrays through ctypes.  It shares nothing with the
CUDA library.

The definitions follow the textbook / PyTorch ``Conv2d`` cross-correlation that
the subject page (clu0's C++/CUDA UNet diffusion, sourcepulse.org project page,
"How It Works" and "Highlighted Details") implies when it speaks of 3x3
convolution kernels forward and backward that aim to match PyTorch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv3x3_oracle.c")
_SRC_UFD = os.path.join(_HERE, "upfirdn2d_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, -O2, no fast-math)."""
    srcs = [_SRC, _SRC_UFD]
    if force or not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(f)
                                                for f in srcs):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
               "-pthread"] + srcs + ["-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_get_threads.restype = ctypes.c_int
        lib.oracle_silu_f64.argtypes = [ctypes.c_double]
        lib.oracle_silu_f64.restype = ctypes.c_double
        lib.oracle_lrelu_f64.argtypes = [ctypes.c_double]
        lib.oracle_lrelu_f64.restype = ctypes.c_double
        lib.oracle_conv3x3_fwd_f64.argtypes = [_dp, _dp, _dp, _dp] + [_i64] * 5 + [ctypes.c_int]
        lib.oracle_conv3x3_fwd_at_f64.argtypes = [_dp, _dp, _dp] + [_i64] * 5 + [ctypes.c_int, _lp, _i64, _dp]
        lib.oracle_act_grad_f64.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.oracle_act_grad_f64.restype = ctypes.c_double
        lib.oracle_conv3x3_dgrad_f64.argtypes = [_dp, _dp, _dp] + [_i64] * 5
        lib.oracle_conv3x3_dgrad_act_f64.argtypes = [_dp, _dp, _dp, ctypes.c_int, _dp] + [_i64] * 5
        lib.oracle_conv3x3_dgrad_act_at_f64.argtypes = ([_dp, _dp, _dp, ctypes.c_int] + [_i64] * 5
                                                        + [_lp, _i64, _dp])
        lib.oracle_conv3x3_dgrad_at_f64.argtypes = [_dp, _dp] + [_i64] * 5 + [_lp, _i64, _dp]
        lib.oracle_conv3x3_wgrad_f64.argtypes = [_dp, _dp, _dp, _dp] + [_i64] * 5
        lib.oracle_conv3x3_wgrad_at_f64.argtypes = [_dp, _dp] + [_i64] * 5 + [_lp, _i64, _dp]
        lib.oracle_conv3x3_dbias_f64.argtypes = [_dp, _dp] + [_i64] * 4
        lib.oracle_conv3x3_fwd_strided_f64.argtypes = [_dp, _dp, _dp, _dp] + [_i64] * 6 + [ctypes.c_int]
        lib.oracle_conv3x3_fwd_strided_at_f64.argtypes = ([_dp, _dp, _dp] + [_i64] * 6
                                                          + [ctypes.c_int, _lp, _i64, _dp])
        lib.oracle_conv3x3_dgrad_strided_f64.argtypes = [_dp, _dp, _dp] + [_i64] * 6
        lib.oracle_conv3x3_dgrad_strided_at_f64.argtypes = [_dp, _dp] + [_i64] * 6 + [_lp, _i64, _dp]
        lib.oracle_conv3x3_wgrad_strided_f64.argtypes = [_dp, _dp, _dp] + [_i64] * 6
        lib.oracle_conv3x3_wgrad_strided_at_f64.argtypes = [_dp, _dp] + [_i64] * 6 + [_lp, _i64, _dp]
        lib.oracle_upfirdn2d_f64.argtypes = [_dp, _dp, _dp] + [_i64] * 12
        lib.oracle_upfirdn2d_at_f64.argtypes = [_dp, _dp] + [_i64] * 12 + [_lp, _i64, _dp]
        lib.oracle_upfirdn2d_out_len.argtypes = [_i64] * 6
        lib.oracle_upfirdn2d_out_len.restype = _i64
        _lib = lib
    return _lib


def _d(a, shape=None):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        a = a.reshape(shape)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def set_threads(n: int) -> None:
    """0 = all online cores (the default)."""
    _load().oracle_set_threads(int(n))


def threads() -> int:
    return int(_load().oracle_get_threads())


def silu(z: float) -> float:
    return float(_load().oracle_silu_f64(float(z)))


def lrelu(z: float) -> float:
    return float(_load().oracle_lrelu_f64(float(z)))


def conv3x3_fwd(x, w, bias=None, act: int = 0):
    """y[n,h,w,k] = act(b[k] + sum_{r,s,c} x[n,h+r-1,w+s-1,c] w[k,r,s,c]); x NHWC, w KRSC.
    act: 0 none, 1 SiLU, 2 leaky ReLU (slope 0.2)."""
    x = _d(x)
    N, H, W, Cin = x.shape
    w = _d(w)
    Cout = w.shape[0]
    assert w.shape == (Cout, 3, 3, Cin), w.shape
    b = None if bias is None else _d(bias, (Cout,))
    y = np.empty((N, H, W, Cout), np.float64)
    _load().oracle_conv3x3_fwd_f64(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, Cin, Cout, H, W, int(act))
    return y


def conv3x3_fwd_at(x, w, bias, act, idx):
    """Forward outputs at the given linear NHWC indices of y."""
    x = _d(x)
    N, H, W, Cin = x.shape
    w = _d(w)
    Cout = w.shape[0]
    b = None if bias is None else _d(bias, (Cout,))
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_fwd_at_f64(_ptr(x), _ptr(w), _ptr(b), N, Cin, Cout, H, W, int(act),
                                      idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


def conv3x3_dgrad(dz, w):
    """dx[n,h,w,c] = sum_{r,s,k} dz[n,h+1-r,w+1-s,k] w[k,r,s,c]."""
    dz = _d(dz)
    N, H, W, Cout = dz.shape
    w = _d(w)
    Cin = w.shape[3]
    assert w.shape == (Cout, 3, 3, Cin), w.shape
    dx = np.empty((N, H, W, Cin), np.float64)
    _load().oracle_conv3x3_dgrad_f64(_ptr(dz), _ptr(w), _ptr(dx), N, Cin, Cout, H, W)
    return dx


def conv3x3_dgrad_at(dz, w, idx):
    dz = _d(dz)
    N, H, W, Cout = dz.shape
    w = _d(w)
    Cin = w.shape[3]
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_dgrad_at_f64(_ptr(dz), _ptr(w), N, Cin, Cout, H, W,
                                        idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


def act_grad(act: int, z: float) -> float:
    """d act / dz at z (act 0 none, 1 SiLU, 2 leaky ReLU)."""
    return float(_load().oracle_act_grad_f64(int(act), float(z)))


def conv3x3_dgrad_act(dz, w, zin, act: int):
    """Gradient with respect to zin when the convolution's input is act(zin):
    act'(zin) * conv3x3_dgrad(dz, w); zin has the layout of the input [N,H,W,Cin]."""
    dz = _d(dz)
    N, H, W, Cout = dz.shape
    w = _d(w)
    Cin = w.shape[3]
    assert w.shape == (Cout, 3, 3, Cin), w.shape
    zin = _d(zin, (N, H, W, Cin))
    dx = np.empty((N, H, W, Cin), np.float64)
    _load().oracle_conv3x3_dgrad_act_f64(_ptr(dz), _ptr(w), _ptr(zin), int(act), _ptr(dx),
                                         N, Cin, Cout, H, W)
    return dx


def conv3x3_dgrad_act_at(dz, w, zin, act: int, idx):
    dz = _d(dz)
    N, H, W, Cout = dz.shape
    w = _d(w)
    Cin = w.shape[3]
    zin = _d(zin, (N, H, W, Cin))
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_dgrad_act_at_f64(_ptr(dz), _ptr(w), _ptr(zin), int(act), N, Cin, Cout,
                                            H, W, idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


# ---------------------------------------------------------------------------
# channel-concatenated input: x = concat(xa, xb) along channels (a UNet up-path
# conv reads its main branch and its skip this way).  The definition is the
# plain convolution of the concatenated tensor; the weight's channels [0, Ca)
# act on xa and [Ca, Ca + Cb) on xb.
# ---------------------------------------------------------------------------
def _cat(xa, xb):
    xa, xb = _d(xa), _d(xb)
    assert xa.shape[:3] == xb.shape[:3], (xa.shape, xb.shape)
    return np.concatenate([xa, xb], axis=-1)


def conv3x3_fwd_cat(xa, xb, w, bias=None, act: int = 0):
    return conv3x3_fwd(_cat(xa, xb), w, bias, act)


def conv3x3_fwd_cat_at(xa, xb, w, bias, act, idx):
    return conv3x3_fwd_at(_cat(xa, xb), w, bias, act, idx)


def conv3x3_dgrad_cat(dz, w, Ca: int):
    """(dxa, dxb): the input gradient split at channel Ca."""
    dx = conv3x3_dgrad(dz, w)
    return np.ascontiguousarray(dx[..., :Ca]), np.ascontiguousarray(dx[..., Ca:])


def conv3x3_wgrad_cat(xa, xb, dz):
    return conv3x3_wgrad(_cat(xa, xb), dz)


def conv3x3_wgrad_cat_at(xa, xb, dz, idx):
    return conv3x3_wgrad_at(_cat(xa, xb), dz, idx)


def conv3x3_wgrad(x, dz):
    """(dw[k,r,s,c], db[k]) = (sum_p dz[p,k] x[p+(r-1,s-1),c], sum_p dz[p,k])."""
    x = _d(x)
    N, H, W, Cin = x.shape
    dz = _d(dz)
    Cout = dz.shape[3]
    assert dz.shape[:3] == (N, H, W)
    dw = np.empty((Cout, 3, 3, Cin), np.float64)
    db = np.empty((Cout,), np.float64)
    _load().oracle_conv3x3_wgrad_f64(_ptr(x), _ptr(dz), _ptr(dw), _ptr(db), N, Cin, Cout, H, W)
    return dw, db


def conv3x3_wgrad_at(x, dz, idx):
    """dw at the given linear KRSC indices (each a full sum over all pixels)."""
    x = _d(x)
    N, H, W, Cin = x.shape
    dz = _d(dz)
    Cout = dz.shape[3]
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_wgrad_at_f64(_ptr(x), _ptr(dz), N, Cin, Cout, H, W,
                                        idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


def conv3x3_dbias(dz):
    dz = _d(dz)
    N, H, W, Cout = dz.shape
    db = np.empty((Cout,), np.float64)
    _load().oracle_conv3x3_dbias_f64(_ptr(dz), _ptr(db), N, Cout, H, W)
    return db


# ---------------------------------------------------------------------------
# strided convolution (stride u, zero padding 1): the UNet's downsampling conv
# ---------------------------------------------------------------------------
def strided_out(length: int, u: int) -> int:
    return (length - 1) // u + 1


def conv3x3_fwd_strided(x, w, bias=None, act: int = 0, u: int = 2):
    """y[n,ho,wo,k] = act(b[k] + sum x[n, u ho + r - 1, u wo + s - 1, c] w[k,r,s,c])."""
    x = _d(x)
    N, H, W, Cin = x.shape
    w = _d(w)
    Cout = w.shape[0]
    assert w.shape == (Cout, 3, 3, Cin), w.shape
    b = None if bias is None else _d(bias, (Cout,))
    y = np.empty((N, strided_out(H, u), strided_out(W, u), Cout), np.float64)
    _load().oracle_conv3x3_fwd_strided_f64(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, Cin, Cout, H, W,
                                           int(u), int(act))
    return y


def conv3x3_fwd_strided_at(x, w, bias, act, u, idx):
    x = _d(x)
    N, H, W, Cin = x.shape
    w = _d(w)
    Cout = w.shape[0]
    b = None if bias is None else _d(bias, (Cout,))
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_fwd_strided_at_f64(_ptr(x), _ptr(w), _ptr(b), N, Cin, Cout, H, W,
                                              int(u), int(act), idx.ctypes.data_as(_lp),
                                              idx.shape[0], _ptr(out))
    return out


def conv3x3_dgrad_strided(dz, w, H: int, W: int, u: int = 2):
    """dx [N,H,W,Cin]: the adjoint of the strided forward applied to dz [N,Ho,Wo,Cout]."""
    dz = _d(dz)
    N, Ho, Wo, Cout = dz.shape
    assert (Ho, Wo) == (strided_out(H, u), strided_out(W, u)), (dz.shape, H, W, u)
    w = _d(w)
    Cin = w.shape[3]
    dx = np.empty((N, H, W, Cin), np.float64)
    _load().oracle_conv3x3_dgrad_strided_f64(_ptr(dz), _ptr(w), _ptr(dx), N, Cin, Cout, H, W,
                                             int(u))
    return dx


def conv3x3_dgrad_strided_at(dz, w, H, W, u, idx):
    dz = _d(dz)
    N, Ho, Wo, Cout = dz.shape
    w = _d(w)
    Cin = w.shape[3]
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_dgrad_strided_at_f64(_ptr(dz), _ptr(w), N, Cin, Cout, H, W, int(u),
                                                idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


def conv3x3_wgrad_strided(x, dz, u: int = 2):
    """(dw [Cout,3,3,Cin], db [Cout]) of the strided convolution."""
    x = _d(x)
    N, H, W, Cin = x.shape
    dz = _d(dz)
    Cout = dz.shape[3]
    assert dz.shape[:3] == (N, strided_out(H, u), strided_out(W, u)), (x.shape, dz.shape)
    out = np.empty(9 * Cin * Cout + Cout, np.float64)
    _load().oracle_conv3x3_wgrad_strided_f64(_ptr(x), _ptr(dz), _ptr(out), N, Cin, Cout, H, W,
                                             int(u))
    return out[:9 * Cin * Cout].reshape(Cout, 3, 3, Cin), out[9 * Cin * Cout:].copy()


def conv3x3_wgrad_strided_at(x, dz, u, idx):
    """dw at linear KRSC indices (an index 9*Cin*Cout + k gives db[k])."""
    x = _d(x)
    N, H, W, Cin = x.shape
    dz = _d(dz)
    Cout = dz.shape[3]
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_conv3x3_wgrad_strided_at_f64(_ptr(x), _ptr(dz), N, Cin, Cout, H, W, int(u),
                                                idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out


# ---------------------------------------------------------------------------
# upfirdn2d: upsample (zeros after each pixel), zero-pad, FIR filter
# (convolution), downsample -- the StyleGAN2 custom-kernel blog's filtered
# up/downsampling (page titled "Dim3 grid calculation code", first paragraph).
# The arithmetic is in upfirdn2d_oracle.c.
# ---------------------------------------------------------------------------
def _pads(pad):
    """(pad_x0, pad_x1, pad_y0, pad_y1) from an int, a pair (x, y) or a 4-tuple."""
    if isinstance(pad, int):
        return pad, pad, pad, pad
    pad = tuple(int(p) for p in pad)
    if len(pad) == 2:
        return pad[0], pad[0], pad[1], pad[1]
    assert len(pad) == 4, pad
    return pad


def upfirdn2d_out_len(length, up, down, p0, p1, k):
    return int(_load().oracle_upfirdn2d_out_len(length, up, down, p0, p1, k))


def upfirdn2d(x, f, up: int = 1, down: int = 1, pad=0):
    """x [N,H,W,C], f [kh,kw]; pad = (pad_x0, pad_x1, pad_y0, pad_y1).  Returns
    y [N,Ho,Wo,C]: every channel upsampled, padded, convolved with f and
    downsampled, in that order."""
    x = _d(x)
    N, H, W, C = x.shape
    f = _d(f)
    kh, kw = f.shape
    px0, px1, py0, py1 = _pads(pad)
    Ho = upfirdn2d_out_len(H, up, down, py0, py1, kh)
    Wo = upfirdn2d_out_len(W, up, down, px0, px1, kw)
    y = np.empty((N, Ho, Wo, C), np.float64)
    _load().oracle_upfirdn2d_f64(_ptr(x), _ptr(f), _ptr(y), N, H, W, C, up, down, px0, px1, py0,
                                 py1, kh, kw)
    return y


def upfirdn2d_at(x, f, up, down, pad, idx):
    """y at the given linear NHWC indices of the output."""
    x = _d(x)
    N, H, W, C = x.shape
    f = _d(f)
    kh, kw = f.shape
    px0, px1, py0, py1 = _pads(pad)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().oracle_upfirdn2d_at_f64(_ptr(x), _ptr(f), N, H, W, C, up, down, px0, px1, py0, py1,
                                    kh, kw, idx.ctypes.data_as(_lp), idx.shape[0], _ptr(out))
    return out
