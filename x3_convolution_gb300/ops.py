"""Torch-tensor convenience layer over the C ABI (allocation and marshalling only).

Tensors are NHWC / KRSC and contiguous; torch only allocates device memory and
supplies the stream.  Each call forwards to one entry point of libconv3x3.so.
"""
from __future__ import annotations

import torch

from . import _lib as L


def _shape(x: torch.Tensor, w: torch.Tensor):
    N, H, W, Cin = x.shape
    Cout = w.shape[0]
    return N, Cin, Cout, H, W


def fwd(x, w, bias=None, act=L.ACT_NONE, out_dtype=L.DT_BF16, path=L.PATH_AUTO, out=None,
        stream=None, z_out=None):
    """y = act(conv3x3(x, w) + bias); x [N,H,W,Cin] bf16, w [Cout,3,3,Cin] bf16.
    With z_out (bf16 [N,H,W,Cout]) the pre-activation is stored there too."""
    N, Cin, Cout, H, W = _shape(x, w)
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, H, W, Cout), dtype=dt, device=x.device)
    if z_out is None:
        L.conv3x3_fwd_ex(x, w, bias, out, N, Cin, Cout, H, W, act, out_dtype, path, stream)
    else:
        L.conv3x3_fwd_save_z(x, w, bias, out, z_out, N, Cin, Cout, H, W, act, out_dtype, path,
                             stream)
    return out


def dgrad(dy, w, out_dtype=L.DT_BF16, path=L.PATH_AUTO, out=None, stream=None, z_in=None,
          act_in=L.ACT_NONE):
    """dx [N,H,W,Cin] from dy [N,H,W,Cout] and w [Cout,3,3,Cin].
    With z_in (bf16 [N,H,W,Cin]) and act_in, returns act_in'(z_in) * dx instead."""
    N, H, W, Cout = dy.shape
    Cin = w.shape[3]
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, H, W, Cin), dtype=dt, device=dy.device)
    if z_in is None:
        L.conv3x3_dgrad_ex(dy, w, out, N, Cin, Cout, H, W, out_dtype, path, stream)
    else:
        L.conv3x3_dgrad_act(dy, w, z_in, act_in, out, N, Cin, Cout, H, W, out_dtype, path, stream)
    return out


def wgrad_workspace(N, Cin, Cout, H, W, path=L.PATH_AUTO, device="cuda"):
    nbytes = L.conv3x3_wgrad_workspace_bytes_ex(N, Cin, Cout, H, W, path)
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device), nbytes


def wgrad(x, dy, with_bias=True, path=L.PATH_AUTO, workspace=None, out=None, stream=None):
    """(dw [Cout,3,3,Cin] fp32, dbias [Cout] fp32)."""
    N, H, W, Cin = x.shape
    Cout = dy.shape[3]
    if workspace is None:
        workspace = wgrad_workspace(N, Cin, Cout, H, W, path, x.device)
    ws, nbytes = workspace
    if out is None:
        dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device=x.device)
        db = torch.empty((Cout,), dtype=torch.float32, device=x.device) if with_bias else None
    else:
        dw, db = out
    L.conv3x3_wgrad_ex(x, dy, dw, db, N, Cin, Cout, H, W, ws, nbytes, path, stream)
    return dw, db


def fwd_f32(x, w, bias=None, act=L.ACT_NONE, stream=None):
    N, Cin, Cout, H, W = _shape(x, w)
    y = torch.empty((N, H, W, Cout), dtype=torch.float32, device=x.device)
    L.conv3x3_fwd_f32(x, w, bias, y, N, Cin, Cout, H, W, act, stream)
    return y


def dgrad_f32(dy, w, stream=None):
    N, H, W, Cout = dy.shape
    Cin = w.shape[3]
    dx = torch.empty((N, H, W, Cin), dtype=torch.float32, device=dy.device)
    L.conv3x3_dgrad_f32(dy, w, dx, N, Cin, Cout, H, W, stream)
    return dx


def wgrad_f32(x, dy, stream=None):
    N, H, W, Cin = x.shape
    Cout = dy.shape[3]
    dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device=x.device)
    db = torch.empty((Cout,), dtype=torch.float32, device=x.device)
    L.conv3x3_wgrad_f32(x, dy, dw, db, N, Cin, Cout, H, W, None, 0, stream)
    return dw, db


# ---------------------------------------------------------------------------
# channel-concatenated input, passed as its two parts
# ---------------------------------------------------------------------------
def fwd_cat(xa, xb, w, bias=None, act=L.ACT_NONE, out_dtype=L.DT_BF16, path=L.PATH_AUTO,
            out=None, z_out=None, stream=None):
    """act(conv3x3(concat(xa, xb), w) + bias) without building the concatenation."""
    N, H, W, Ca = xa.shape
    Cin, Cout = Ca + xb.shape[3], w.shape[0]
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, H, W, Cout), dtype=dt, device=xa.device)
    L.conv3x3_fwd_cat(xa, xb, Ca, w, bias, out, z_out, N, Cin, Cout, H, W, act, out_dtype, path,
                      stream)
    return out


def dgrad_cat(dy, w, Ca, out_dtype=L.DT_BF16, path=L.PATH_AUTO, out=None, za_in=None, zb_in=None,
              act_in=L.ACT_NONE, stream=None):
    """(dxa, dxb): the input gradient of a conv over concat(xa, xb), split at channel Ca."""
    N, H, W, Cout = dy.shape
    Cin = w.shape[3]
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = (torch.empty((N, H, W, Ca), dtype=dt, device=dy.device),
               torch.empty((N, H, W, Cin - Ca), dtype=dt, device=dy.device))
    dxa, dxb = out
    L.conv3x3_dgrad_cat(dy, w, dxa, dxb, Ca, za_in, zb_in, act_in, N, Cin, Cout, H, W, out_dtype,
                        path, stream)
    return dxa, dxb


def wgrad_cat(xa, xb, dy, with_bias=True, path=L.PATH_AUTO, out=None, stream=None):
    """(dw [Cout,3,3,Cin] fp32, dbias [Cout] fp32) of a conv over concat(xa, xb)."""
    N, H, W, Ca = xa.shape
    Cin, Cout = Ca + xb.shape[3], dy.shape[3]
    nbytes = L.conv3x3_wgrad_cat_workspace_bytes(N, Cin, Ca, Cout, H, W, path)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=xa.device)
    if out is None:
        dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device=xa.device)
        db = torch.empty((Cout,), dtype=torch.float32, device=xa.device) if with_bias else None
    else:
        dw, db = out
    L.conv3x3_wgrad_cat(xa, xb, Ca, dy, dw, db, N, Cin, Cout, H, W, ws, nbytes, path, stream)
    return dw, db


# ---------------------------------------------------------------------------
# strided (downsampling) convolution
# ---------------------------------------------------------------------------
def strided_out(length, stride):
    return (length - 1) // stride + 1


def fwd_strided(x, w, bias=None, stride=2, act=L.ACT_NONE, out_dtype=L.DT_BF16,
                path=L.PATH_AUTO, out=None, z_out=None, stream=None):
    """y [N, Ho, Wo, Cout] of the stride-`stride`, pad-1 3x3 convolution."""
    N, Cin, Cout, H, W = _shape(x, w)
    Ho, Wo = strided_out(H, stride), strided_out(W, stride)
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, Ho, Wo, Cout), dtype=dt, device=x.device)
    L.conv3x3_fwd_strided(x, w, bias, out, z_out, N, Cin, Cout, H, W, stride, act, out_dtype, path,
                          stream)
    return out


def dgrad_strided(dy, w, H, W, stride=2, out_dtype=L.DT_BF16, path=L.PATH_AUTO, out=None,
                  z_in=None, act_in=L.ACT_NONE, stream=None):
    """dx [N, H, W, Cin] from dy [N, Ho, Wo, Cout]."""
    N = dy.shape[0]
    Cout, Cin = w.shape[0], w.shape[3]
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, H, W, Cin), dtype=dt, device=dy.device)
    L.conv3x3_dgrad_strided(dy, w, out, z_in, act_in, N, Cin, Cout, H, W, stride, out_dtype, path,
                            stream)
    return out


def wgrad_strided(x, dy, stride=2, with_bias=True, path=L.PATH_AUTO, out=None, stream=None):
    N, H, W, Cin = x.shape
    Cout = dy.shape[3]
    nbytes = L.conv3x3_wgrad_strided_workspace_bytes(N, Cin, Cout, H, W, stride, path)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    if out is None:
        dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device=x.device)
        db = torch.empty((Cout,), dtype=torch.float32, device=x.device) if with_bias else None
    else:
        dw, db = out
    L.conv3x3_wgrad_strided(x, dy, dw, db, N, Cin, Cout, H, W, stride, ws, nbytes, path, stream)
    return dw, db


def upfirdn2d(x, f, up=1, down=1, pad=(0, 0, 0, 0), out_dtype=L.DT_BF16, out=None, stream=None):
    """Filtered resampling of x [N,H,W,C] bf16 with the host filter f [kh,kw]:
    upsample (zeros after each pixel), zero-pad (pad_x0, pad_x1, pad_y0,
    pad_y1), convolve with f, keep every down-th pixel.  Returns y [N,Ho,Wo,C]."""
    import numpy as np
    N, H, W, C = x.shape
    f = np.asarray(f, dtype=np.float32)
    kh, kw = f.shape
    px0, px1, py0, py1 = pad
    Ho = L.upfirdn2d_out_size(H, up, down, py0, py1, kh)
    Wo = L.upfirdn2d_out_size(W, up, down, px0, px1, kw)
    if out is None:
        dt = torch.float32 if out_dtype == L.DT_F32 else torch.bfloat16
        out = torch.empty((N, max(Ho, 1), max(Wo, 1), C), dtype=dt, device=x.device)
    L.upfirdn2d(x, f, out, N, C, H, W, up, down, px0, px1, py0, py1, kh, kw, out_dtype, stream)
    return out
