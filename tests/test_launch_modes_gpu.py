"""The launch modes the benchmark step uses give the same bits as plain calls.

* A CUDA-graph replay of fwd / dgrad / wgrad.
* Two wgrad calls running at once on two streams, each with its own split-K
  workspace: a wgrad reads only its layer's x and dy, and its reduction is in a
  fixed order.
* Launches without programmatic dependent launch (CONV3X3_PDL=0, read once per
  process, so that side runs in a child process).

Shapes pick each kernel family: the transposed 128-channel tile (64x64, 128
channels, batch 16), the CTA-pair dgrad (32x32, 256 channels, batch 40: enough pair
tiles for two rounds) and the 8-channel stem kernels.
"""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys

import pytest
import torch

import synth
from x3_convolution_gb300 import _lib as L
from x3_convolution_gb300 import ops

from gpu_util import to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# N, Cin, Cout, H, W
SHAPES = [(16, 128, 128, 64, 64), (40, 256, 256, 32, 32), (4, 8, 128, 64, 64)]


def _inputs(shape, seed=3):
    N, Cin, Cout, H, W = shape
    t = synth.make_tensors(synth.Layer("modes", N, Cin, Cout, H, W, act=1), seed=seed)
    return to_dev_bf16(t.x), to_dev_bf16(t.w), to_dev_f32(t.bias), to_dev_bf16(t.dy)


def _digest(tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def _plain(shape):
    x, w, b, dy = _inputs(shape)
    y = ops.fwd(x, w, b, act=L.ACT_SILU)
    dx = ops.dgrad(dy, w)
    dw, db = ops.wgrad(x, dy)
    torch.cuda.synchronize()
    assert L.conv3x3_device_status() == L.OK
    return y, dx, dw, db


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_graph_replay_bit_identical(shape):
    ref = _plain(shape)
    x, w, b, dy = _inputs(shape)
    N, Cin, Cout, H, W = shape
    y = torch.empty_like(ref[0])
    dx = torch.empty_like(ref[1])
    dw, db = torch.empty_like(ref[2]), torch.empty_like(ref[3])
    ws = ops.wgrad_workspace(N, Cin, Cout, H, W)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first calls outside capture (one-time set-up)
        ops.fwd(x, w, b, act=L.ACT_SILU, out=y, stream=s)
        ops.dgrad(dy, w, out=dx, stream=s)
        ops.wgrad(x, dy, workspace=ws, out=(dw, db), stream=s)
    torch.cuda.synchronize()
    for t in (y, dx, dw, db):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.fwd(x, w, b, act=L.ACT_SILU, out=y, stream=s)
        ops.dgrad(dy, w, out=dx, stream=s)
        ops.wgrad(x, dy, workspace=ws, out=(dw, db), stream=s)
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert L.conv3x3_device_status() == L.OK
        for got, want in zip((y, dx, dw, db), ref):
            assert torch.equal(got, want)


def test_concurrent_wgrad_streams_bit_identical():
    a, b = SHAPES[0], SHAPES[1]
    xa, _, _, dya = _inputs(a, seed=5)
    xb, _, _, dyb = _inputs(b, seed=6)
    ra = ops.wgrad(xa, dya)
    rb = ops.wgrad(xb, dyb)
    torch.cuda.synchronize()
    wsa = ops.wgrad_workspace(*a)
    wsb = ops.wgrad_workspace(*b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        ga = ops.wgrad(xa, dya, workspace=wsa, stream=s1)
        gb = ops.wgrad(xb, dyb, workspace=wsb, stream=s2)
        outs.append((ga, gb))
    torch.cuda.synchronize()
    assert L.conv3x3_device_status() == L.OK
    for ga, gb in outs:
        assert torch.equal(ga[0], ra[0]) and torch.equal(ga[1], ra[1])
        assert torch.equal(gb[0], rb[0]) and torch.equal(gb[1], rb[1])


_CHILD = r"""
import hashlib, sys
import torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_launch_modes_gpu as m
for shape in m.SHAPES:
    print(m._digest(m._plain(shape)))
"""


def test_without_programmatic_dependent_launch_bit_identical():
    want = [_digest(_plain(shape)) for shape in SHAPES]
    env = dict(os.environ, CONV3X3_PDL="0")
    code = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    got = r.stdout.split()
    assert got == want
