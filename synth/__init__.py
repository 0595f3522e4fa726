"""Seeded synthetic inputs for the 3x3 convolution workloads.

Shared by the tests and the benchmark; holds none of the convolution's
arithmetic.  ``synth.c`` turns (stream, index) into N(0, std^2) float32 samples
(splitmix64 + Box-Muller); this module names the workloads and the tensors
they draw.

The workloads stand in for the 64x64 ImageNet diffusion UNet that the subject
page trains (clu0's C++/CUDA UNet diffusion, sourcepulse.org project page,
"Quick Start & Requirements": ImageNet 64x64 data); no dataset or trained
weight is used anywhere.

Stream ids: (seed << 32) | (layer << 8) | tensor, tensor = 0 x, 1 w, 2 bias, 3 dy,
4 z_in (the pre-activation of the layer that produced x, for the fused backward
through that activation; N(0, 1), laid out like x).
Distributions: x, dy ~ N(0, 1); w ~ N(0, 2 / (9 * Cin_real)) (Kaiming normal with
the real fan-in); bias ~ N(0, 0.02^2).  bf16 workloads round each float32 sample
to bf16 round-to-nearest-even; the stem's three image channels are zero-padded to
eight in both x and w (and therefore in dy's gradient targets dx, dw).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

X, WT, BIAS, DY, ZIN = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                         ctypes.POINTER(ctypes.c_float)]
        _lib = lib
    return _lib


def stream_id(seed: int, layer: int, tensor: int) -> int:
    return ((int(seed) & 0xFFFFFFFF) << 32) | ((int(layer) & 0xFFFFFF) << 8) | (int(tensor) & 0xFF)


def normal(stream: int, shape, std: float = 1.0) -> np.ndarray:
    """float32 array of the given shape: std * N(0,1) from one counter-based stream."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, np.float32)
    if n:
        _load().synth_normal_f32(ctypes.c_uint64(stream), n, float(std),
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out.reshape(shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), still as float32."""
    return (bf16_bits(a).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    Cin: int          # channels as laid out in memory (stem: padded to 8)
    Cout: int
    H: int
    W: int
    act: int = 1      # 0 none, 1 SiLU (fwd epilogue)
    cin_real: int = 0  # channels that carry data (stem: 3); 0 means Cin
    dtype: str = "bf16"
    cat_a: int = 0     # up-path conv1: x = concat(main, skip) and main has cat_a channels; 0 = one tensor
    stride: int = 1    # 2: downsampling conv (y and dy on the (H-1)//2+1 x (W-1)//2+1 grid)

    @property
    def P(self) -> int:
        return self.N * self.H * self.W

    @property
    def Ho(self) -> int:
        return (self.H - 1) // self.stride + 1

    @property
    def Wo(self) -> int:
        return (self.W - 1) // self.stride + 1

    @property
    def Po(self) -> int:
        return self.N * self.Ho * self.Wo

    @property
    def real_cin(self) -> int:
        return self.cin_real or self.Cin

    def flops_per_pass(self, padded: bool = False) -> int:
        """2 * N*Ho*Wo * Cin * Cout * 9 (real Cin unless padded=True)."""
        cin = self.Cin if padded else self.real_cin
        return 2 * self.Po * cin * self.Cout * 9


@dataclass
class Tensors:
    """float32 arrays holding exactly the values each side computes with."""
    x: np.ndarray
    w: np.ndarray
    bias: np.ndarray
    dy: np.ndarray
    layer: Layer = field(repr=False, default=None)


def make_tensors(layer: Layer, seed: int = 0, index: int = 0, round_bf16: bool | None = None) -> Tensors:
    """Seeded x (NHWC), w (KRSC), bias, dy (NHWC) for one layer."""
    L = layer
    rb = (L.dtype == "bf16") if round_bf16 is None else round_bf16
    cr = L.real_cin
    x = normal(stream_id(seed, index, X), (L.N, L.H, L.W, cr), 1.0)
    w = normal(stream_id(seed, index, WT), (L.Cout, 3, 3, cr), math.sqrt(2.0 / (9 * cr)))
    b = normal(stream_id(seed, index, BIAS), (L.Cout,), 0.02)
    dy = normal(stream_id(seed, index, DY), (L.N, L.Ho, L.Wo, L.Cout), 1.0)
    if cr != L.Cin:  # zero-pad the channel dimension (stem: 3 -> 8)
        xp = np.zeros((L.N, L.H, L.W, L.Cin), np.float32)
        xp[..., :cr] = x
        wp = np.zeros((L.Cout, 3, 3, L.Cin), np.float32)
        wp[..., :cr] = w
        x, w = xp, wp
    if rb:
        x, w, dy = bf16_round(x), bf16_round(w), bf16_round(dy)
    return Tensors(x=x, w=w, bias=b, dy=dy, layer=L)


def make_zin(layer: Layer, seed: int = 0, index: int = 0, round_bf16: bool | None = None) -> np.ndarray:
    """Seeded z_in [N, H, W, Cin] ~ N(0, 1): the input's pre-activation."""
    L = layer
    rb = (L.dtype == "bf16") if round_bf16 is None else round_bf16
    z = normal(stream_id(seed, index, ZIN), (L.N, L.H, L.W, L.Cin), 1.0)
    return bf16_round(z) if rb else z


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
TINY = Layer("tiny", 2, 64, 64, 32, 32, act=0, dtype="f32")
STEM = Layer("stem", 64, 8, 128, 64, 64, act=1, cin_real=3)
L1 = Layer("l1", 64, 128, 128, 64, 64, act=1)
L2 = Layer("l2", 64, 256, 256, 32, 32, act=1)
L3 = Layer("l3", 64, 384, 384, 16, 16, act=1)
# the UNet's deepest level (not a gate config): 512 channels at 8x8
L4 = Layer("l4", 64, 512, 512, 8, 8, act=1)


def unet_stack(N: int = 64, base: int = 128, mult=(1, 2, 3, 4), res0: int = 64,
               blocks: int = 2) -> list[Layer]:
    """The 3x3 convs of the UNet's down and up resblocks (two convs per resblock).

    Down path, level l (channels c_l = base*mult[l], resolution res0 / 2^l): each
    resblock is conv(c_in -> c_l), conv(c_l -> c_l) and pushes one skip of c_l
    channels.  Up path, levels from the deepest up: each resblock is
    conv(main + skip -> c_l), conv(c_l -> c_l), popping skips in reverse order;
    the main branch enters the deepest level with its own channel count and then
    carries the level below's.  With the defaults: 32 convs, up-path Cin =
    1024, 1024 @8x8; 896, 768 @16x16; 640, 512 @32x32; 384, 256 @64x64.
    """
    layers: list[Layer] = []
    skips: list[int] = []
    c_in = base
    for l, m in enumerate(mult):
        c, r = base * m, res0 >> l
        for b in range(blocks):
            layers.append(Layer(f"down{l}.rb{b}.conv1", N, c_in, c, r, r))
            layers.append(Layer(f"down{l}.rb{b}.conv2", N, c, c, r, r))
            skips.append(c)
            c_in = c
    main = c_in
    for l in reversed(range(len(mult))):
        c, r = base * mult[l], res0 >> l
        for b in range(blocks):
            s = skips.pop()
            layers.append(Layer(f"up{l}.rb{b}.conv1", N, main + s, c, r, r, cat_a=main))
            layers.append(Layer(f"up{l}.rb{b}.conv2", N, c, c, r, r))
            main = c
    return layers


STACK = unet_stack()

# The UNet's downsampling convs between levels (stride 2, channels kept):
# 128 @64x64 -> 32x32, 256 @32x32 -> 16x16, 384 @16x16 -> 8x8.
DOWNSAMPLE = [Layer(f"down{l}.downsample", 64, c, c, r, r, stride=2)
              for l, (c, r) in enumerate([(128, 64), (256, 32), (384, 16)])]

# The benchmark's training-step sweep: the stem conv followed by the 32 resblock convs.
UNET_STEP = [STEM] + STACK

CONFIGS = {"tiny": [TINY], "stem": [STEM], "l1": [L1], "l2": [L2], "l3": [L3], "l4": [L4], "stack": STACK,
           "unet": UNET_STEP, "downsample": DOWNSAMPLE}


# ---------------------------------------------------------------------------
# filtered resampling (upfirdn2d) between the UNet's levels
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Resample:
    """One upfirdn2d op: x [N, H, W, C] resampled by `up` / `down` with the
    binomial [1,3,3,1] (x) [1,3,3,1] / 64 filter (times up^2 when upsampling,
    so that a constant keeps its value) and pads (pad_x0, pad_x1, pad_y0,
    pad_y1) that make the output exactly 2x or 1/2x the input."""
    name: str
    N: int
    C: int
    H: int
    W: int
    up: int = 1
    down: int = 1
    pad: tuple = (0, 0, 0, 0)

    def filter(self) -> np.ndarray:
        a = np.array([1.0, 3.0, 3.0, 1.0], np.float64)
        return (np.outer(a, a) / 64.0 * self.up * self.up).astype(np.float32)

    @property
    def Ho(self) -> int:
        return (self.H * self.up + self.pad[2] + self.pad[3] - 4) // self.down + 1

    @property
    def Wo(self) -> int:
        return (self.W * self.up + self.pad[0] + self.pad[1] - 4) // self.down + 1

    def bytes(self) -> int:
        """Algorithmic HBM bytes: x read once, y written once (bf16)."""
        return 2 * self.C * self.N * (self.H * self.W + self.Ho * self.Wo)


def make_resample_input(op: Resample, seed: int = 0, index: int = 0) -> np.ndarray:
    """Seeded x [N, H, W, C] ~ N(0, 1), rounded to bf16."""
    return bf16_round(normal(stream_id(seed, 64 + index, X), (op.N, op.H, op.W, op.C), 1.0))


# The resampling between the UNet's levels (base 128, multipliers 1,2,3,4,
# 64 -> 8 and back), batch 64: 2x downsampling (pads 1, 1) on the way down,
# 2x upsampling (pads 2, 1) on the way up.
UPFIRDN2D = ([Resample(f"down{l}.blur_down", 64, c, r, r, down=2, pad=(1, 1, 1, 1))
              for l, (c, r) in enumerate([(128, 64), (256, 32), (384, 16)])]
             + [Resample(f"up{l}.blur_up", 64, c, r, r, up=2, pad=(2, 1, 2, 1))
                for l, (c, r) in zip((3, 2, 1), [(512, 8), (384, 16), (256, 32)])])
