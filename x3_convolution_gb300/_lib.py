"""ctypes binding to libconv3x3.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/conv3x3.h``) and does nothing but turn tensors into pointers and the
returned status into an exception.  All arithmetic happens in the library's
CUDA kernels; if the library is missing this module raises instead of falling
back to anything.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libconv3x3.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(6)
ACT_NONE, ACT_SILU, ACT_LRELU = 0, 1, 2
DT_BF16, DT_F32 = 0, 1
PATH_AUTO, PATH_TENSOR, PATH_SIMT = 0, 1, 2

_lib = None

_vp, _i, _sz, _ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_ulonglong

_SIGS = {
    "conv3x3_fwd": ([_vp, _vp, _vp, _vp] + [_i] * 6 + [_vp], _i),
    "conv3x3_dgrad": ([_vp, _vp, _vp] + [_i] * 5 + [_vp], _i),
    "conv3x3_wgrad": ([_vp, _vp, _vp, _vp] + [_i] * 5 + [_vp, _sz, _vp], _i),
    "conv3x3_wgrad_workspace_bytes": ([_i] * 5, _sz),
    "conv3x3_fwd_ex": ([_vp, _vp, _vp, _vp] + [_i] * 8 + [_vp], _i),
    "conv3x3_dgrad_ex": ([_vp, _vp, _vp] + [_i] * 7 + [_vp], _i),
    "conv3x3_wgrad_ex": ([_vp, _vp, _vp, _vp] + [_i] * 5 + [_vp, _sz, _i, _vp], _i),
    "conv3x3_wgrad_workspace_bytes_ex": ([_i] * 6, _sz),
    "conv3x3_fwd_f32": ([_vp, _vp, _vp, _vp] + [_i] * 6 + [_vp], _i),
    "conv3x3_dgrad_f32": ([_vp, _vp, _vp] + [_i] * 5 + [_vp], _i),
    "conv3x3_wgrad_f32": ([_vp, _vp, _vp, _vp] + [_i] * 5 + [_vp, _sz, _vp], _i),
    "conv3x3_device_status": ([_vp], _i),
    "conv3x3_selftest_wait_timeout": ([_ull, _vp], _i),
    "conv3x3_status_string": ([_i], ctypes.c_char_p),
    "conv3x3_auto_path": ([_i] * 6, _i),
    "conv3x3_wgrad_noalloc": ([_vp, _vp, _vp, _vp] + [_i] * 5 + [_vp], _i),
    "conv3x3_fwd_save_z": ([_vp, _vp, _vp, _vp, _vp] + [_i] * 8 + [_vp], _i),
    "conv3x3_dgrad_act": ([_vp, _vp, _vp, _i, _vp] + [_i] * 7 + [_vp], _i),
    "conv3x3_fwd_cat": ([_vp, _vp, _i, _vp, _vp, _vp, _vp] + [_i] * 8 + [_vp], _i),
    "conv3x3_dgrad_cat": ([_vp, _vp, _vp, _vp, _i, _vp, _vp, _i] + [_i] * 7 + [_vp], _i),
    "conv3x3_wgrad_cat": ([_vp, _vp, _i, _vp, _vp, _vp] + [_i] * 5 + [_vp, _sz, _i, _vp], _i),
    "conv3x3_wgrad_cat_workspace_bytes": ([_i] * 7, _sz),
    "conv3x3_fwd_strided": ([_vp, _vp, _vp, _vp, _vp] + [_i] * 9 + [_vp], _i),
    "conv3x3_dgrad_strided": ([_vp, _vp, _vp, _vp, _i] + [_i] * 8 + [_vp], _i),
    "conv3x3_wgrad_strided": ([_vp, _vp, _vp, _vp] + [_i] * 6 + [_vp, _sz, _i, _vp], _i),
    "conv3x3_wgrad_strided_workspace_bytes": ([_i] * 7, _sz),
    "upfirdn2d": ([_vp, ctypes.POINTER(ctypes.c_float), _vp] + [_i] * 13 + [_vp], _i),
    "upfirdn2d_out_size": ([_i] * 6, _i),
}

WGRAD_NOALLOC_MAX_BYTES = 64 << 20


class Conv3x3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))
        self.status = status


def load():
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libconv3x3.so not built: run __graft_entry__.build() or "
                              "python x3_convolution_gb300/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().conv3x3_status_string(int(status)).decode()


def _p(t):
    """Device pointer of a tensor (or an int address / None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str) -> int:
    if rc != OK:
        raise Conv3x3Error(rc, what)
    return rc


def conv3x3_fwd(x, w, bias, y, N, Cin, Cout, H, W, act=ACT_NONE, stream=None):
    return _check(load().conv3x3_fwd(_p(x), _p(w), _p(bias), _p(y), N, Cin, Cout, H, W, act,
                                     _stream(stream)), "conv3x3_fwd")


def conv3x3_dgrad(dy, w, dx, N, Cin, Cout, H, W, stream=None):
    return _check(load().conv3x3_dgrad(_p(dy), _p(w), _p(dx), N, Cin, Cout, H, W, _stream(stream)),
                  "conv3x3_dgrad")


def conv3x3_wgrad(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes, stream=None):
    return _check(load().conv3x3_wgrad(_p(x), _p(dy), _p(dw), _p(dbias), N, Cin, Cout, H, W,
                                       _p(workspace), int(workspace_bytes), _stream(stream)),
                  "conv3x3_wgrad")


def conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W) -> int:
    return int(load().conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W))


def conv3x3_fwd_ex(x, w, bias, y, N, Cin, Cout, H, W, act, out_dtype, path, stream=None):
    return _check(load().conv3x3_fwd_ex(_p(x), _p(w), _p(bias), _p(y), N, Cin, Cout, H, W, act,
                                        out_dtype, path, _stream(stream)), "conv3x3_fwd_ex")


def conv3x3_dgrad_ex(dy, w, dx, N, Cin, Cout, H, W, out_dtype, path, stream=None):
    return _check(load().conv3x3_dgrad_ex(_p(dy), _p(w), _p(dx), N, Cin, Cout, H, W, out_dtype,
                                          path, _stream(stream)), "conv3x3_dgrad_ex")


def conv3x3_fwd_save_z(x, w, bias, y, z, N, Cin, Cout, H, W, act, out_dtype, path, stream=None):
    return _check(load().conv3x3_fwd_save_z(_p(x), _p(w), _p(bias), _p(y), _p(z), N, Cin, Cout, H,
                                            W, act, out_dtype, path, _stream(stream)),
                  "conv3x3_fwd_save_z")


def conv3x3_dgrad_act(dy, w, z_in, act_in, dx, N, Cin, Cout, H, W, out_dtype, path, stream=None):
    return _check(load().conv3x3_dgrad_act(_p(dy), _p(w), _p(z_in), act_in, _p(dx), N, Cin, Cout,
                                           H, W, out_dtype, path, _stream(stream)),
                  "conv3x3_dgrad_act")


def conv3x3_fwd_cat(xa, xb, Ca, w, bias, y, z, N, Cin, Cout, H, W, act, out_dtype, path,
                    stream=None):
    return _check(load().conv3x3_fwd_cat(_p(xa), _p(xb), Ca, _p(w), _p(bias), _p(y), _p(z), N, Cin,
                                         Cout, H, W, act, out_dtype, path, _stream(stream)),
                  "conv3x3_fwd_cat")


def conv3x3_dgrad_cat(dy, w, dxa, dxb, Ca, za_in, zb_in, act_in, N, Cin, Cout, H, W, out_dtype,
                      path, stream=None):
    return _check(load().conv3x3_dgrad_cat(_p(dy), _p(w), _p(dxa), _p(dxb), Ca, _p(za_in),
                                           _p(zb_in), act_in, N, Cin, Cout, H, W, out_dtype, path,
                                           _stream(stream)), "conv3x3_dgrad_cat")


def conv3x3_wgrad_cat(xa, xb, Ca, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes,
                      path, stream=None):
    return _check(load().conv3x3_wgrad_cat(_p(xa), _p(xb), Ca, _p(dy), _p(dw), _p(dbias), N, Cin,
                                           Cout, H, W, _p(workspace), int(workspace_bytes), path,
                                           _stream(stream)), "conv3x3_wgrad_cat")


def conv3x3_wgrad_cat_workspace_bytes(N, Cin, Ca, Cout, H, W, path) -> int:
    return int(load().conv3x3_wgrad_cat_workspace_bytes(N, Cin, Ca, Cout, H, W, path))


def conv3x3_fwd_strided(x, w, bias, y, z, N, Cin, Cout, H, W, stride, act, out_dtype, path,
                        stream=None):
    return _check(load().conv3x3_fwd_strided(_p(x), _p(w), _p(bias), _p(y), _p(z), N, Cin, Cout, H,
                                             W, stride, act, out_dtype, path, _stream(stream)),
                  "conv3x3_fwd_strided")


def conv3x3_dgrad_strided(dy, w, dx, z_in, act_in, N, Cin, Cout, H, W, stride, out_dtype, path,
                          stream=None):
    return _check(load().conv3x3_dgrad_strided(_p(dy), _p(w), _p(dx), _p(z_in), act_in, N, Cin,
                                               Cout, H, W, stride, out_dtype, path,
                                               _stream(stream)), "conv3x3_dgrad_strided")


def conv3x3_wgrad_strided(x, dy, dw, dbias, N, Cin, Cout, H, W, stride, workspace,
                          workspace_bytes, path, stream=None):
    return _check(load().conv3x3_wgrad_strided(_p(x), _p(dy), _p(dw), _p(dbias), N, Cin, Cout, H,
                                               W, stride, _p(workspace), int(workspace_bytes),
                                               path, _stream(stream)), "conv3x3_wgrad_strided")


def conv3x3_wgrad_strided_workspace_bytes(N, Cin, Cout, H, W, stride, path) -> int:
    return int(load().conv3x3_wgrad_strided_workspace_bytes(N, Cin, Cout, H, W, stride, path))


def conv3x3_wgrad_ex(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes, path,
                     stream=None):
    return _check(load().conv3x3_wgrad_ex(_p(x), _p(dy), _p(dw), _p(dbias), N, Cin, Cout, H, W,
                                          _p(workspace), int(workspace_bytes), path,
                                          _stream(stream)), "conv3x3_wgrad_ex")


def conv3x3_wgrad_workspace_bytes_ex(N, Cin, Cout, H, W, path) -> int:
    return int(load().conv3x3_wgrad_workspace_bytes_ex(N, Cin, Cout, H, W, path))


def conv3x3_fwd_f32(x, w, bias, y, N, Cin, Cout, H, W, act=ACT_NONE, stream=None):
    return _check(load().conv3x3_fwd_f32(_p(x), _p(w), _p(bias), _p(y), N, Cin, Cout, H, W, act,
                                         _stream(stream)), "conv3x3_fwd_f32")


def conv3x3_dgrad_f32(dy, w, dx, N, Cin, Cout, H, W, stream=None):
    return _check(load().conv3x3_dgrad_f32(_p(dy), _p(w), _p(dx), N, Cin, Cout, H, W,
                                           _stream(stream)), "conv3x3_dgrad_f32")


def conv3x3_wgrad_f32(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace=None, workspace_bytes=0,
                      stream=None):
    return _check(load().conv3x3_wgrad_f32(_p(x), _p(dy), _p(dw), _p(dbias), N, Cin, Cout, H, W,
                                           _p(workspace), int(workspace_bytes), _stream(stream)),
                  "conv3x3_wgrad_f32")


def conv3x3_device_status(stream=None) -> int:
    return int(load().conv3x3_device_status(_stream(stream)))


def conv3x3_selftest_wait_timeout(limit_ns, stream=None):
    return _check(load().conv3x3_selftest_wait_timeout(int(limit_ns), _stream(stream)),
                  "conv3x3_selftest_wait_timeout")


def conv3x3_auto_path(pass_, N, Cin, Cout, H, W) -> int:
    return int(load().conv3x3_auto_path(pass_, N, Cin, Cout, H, W))


def conv3x3_status_string(status) -> str:
    return status_string(status)


def conv3x3_wgrad_noalloc(x, dy, dw, dbias, N, Cin, Cout, H, W, stream=None):
    """conv3x3_wgrad for callers that cannot allocate device memory: the split-K
    scratch comes from a fixed 64 MiB array inside the library (see the C header
    for the sharing rules)."""
    return _check(load().conv3x3_wgrad_noalloc(_p(x), _p(dy), _p(dw), _p(dbias), N, Cin, Cout, H, W,
                                               _stream(stream)), "conv3x3_wgrad_noalloc")


def _host_f32(a):
    """A host fp32 array (filter taps) as a ctypes pointer, and its keep-alive."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float32).reshape(-1))
    return arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), arr


def upfirdn2d(x, f, y, N, C, H, W, up, down, pad_x0, pad_x1, pad_y0, pad_y1, kh, kw,
              out_dtype=DT_BF16, stream=None):
    fp, keep = _host_f32(f)
    rc = load().upfirdn2d(_p(x), fp, _p(y), N, C, H, W, up, down, pad_x0, pad_x1, pad_y0, pad_y1,
                          kh, kw, out_dtype, _stream(stream))
    del keep
    return _check(rc, "upfirdn2d")


def upfirdn2d_out_size(length, up, down, pad0, pad1, k) -> int:
    return int(load().upfirdn2d_out_size(length, up, down, pad0, pad1, k))
