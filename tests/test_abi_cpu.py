"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from x3_convolution_gb300 import build as b
    b.build()
    from x3_convolution_gb300 import _lib
    return _lib.load()


def declared_functions():
    """Every function declared in include/*.h."""
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            src = open(os.path.join(INCLUDE, h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b((?:conv3x3|upfirdn2d)\w*)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["conv3x3_fwd", "conv3x3_dgrad", "conv3x3_wgrad", "conv3x3_wgrad_workspace_bytes",
              "conv3x3_fwd_f32", "conv3x3_dgrad_f32", "conv3x3_wgrad_f32",
              "conv3x3_device_status", "conv3x3_status_string"]:
        assert n in names


def test_upfirdn2d_is_declared_and_validates_without_a_gpu(lib):
    assert "upfirdn2d" in declared_functions() and "upfirdn2d_out_size" in declared_functions()
    assert lib.upfirdn2d_out_size(64, 2, 1, 2, 1, 4) == 128
    assert lib.upfirdn2d_out_size(64, 1, 2, 1, 1, 4) == 32
    assert lib.upfirdn2d_out_size(64, 9, 1, 0, 0, 4) == 0     # factor beyond the limit
    assert lib.upfirdn2d_out_size(64, 1, 1, -1, 0, 4) == 0    # cropping is not a pad
    assert lib.upfirdn2d_out_size(2, 1, 1, 0, 0, 4) == 0      # kernel longer than the plane
    f = (ctypes.c_float * 16)(*([1.0 / 16] * 16))
    ok = (ALIGNED, f, ALIGNED, 2, 64, 8, 8, 1, 2, 1, 1, 1, 1, 4, 4, 0, None)
    bad = [dict(C=12), dict(C=0), dict(up=0), dict(down=9), dict(kh=9), dict(px0=-1),
           dict(dtype=2), dict(x=ALIGNED + 4), dict(f=None)]
    keys = ["x", "f", "y", "N", "C", "H", "W", "up", "down", "px0", "px1", "py0", "py1", "kh", "kw",
            "dtype", "stream"]
    for b in bad:
        a = dict(zip(keys, ok))
        a.update(b)
        assert lib.upfirdn2d(*[a[k] for k in keys]) == 1, b


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_names_match_the_c_entry_points(lib):
    from x3_convolution_gb300 import _lib
    for n in declared_functions():
        assert callable(getattr(_lib, n)), n


def test_status_strings(lib):
    from x3_convolution_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "invalid" in _lib.status_string(1)
    assert "timed out" in _lib.status_string(4)
    assert _lib.status_string(99) == "unknown status"


ALIGNED = 1 << 20  # a fake 16-byte-aligned address; never dereferenced (validation fails first)


@pytest.mark.parametrize("args", [
    dict(N=0, Cin=64, Cout=64, H=8, W=8),     # empty batch
    dict(N=1, Cin=3, Cout=64, H=8, W=8),      # Cin not a multiple of 8
    dict(N=1, Cin=64, Cout=12, H=8, W=8),     # Cout not a multiple of 8
    dict(N=1, Cin=64, Cout=64, H=0, W=8),     # empty image
    dict(N=1, Cin=64, Cout=64, H=70000, W=1),  # H beyond 16 bits
    dict(N=1 << 20, Cin=1024, Cout=64, H=64, W=64),  # tensor beyond 2^31 elements
])
def test_bad_shapes_are_rejected_without_a_gpu(lib, args):
    a = [args[k] for k in ("N", "Cin", "Cout", "H", "W")]
    assert lib.conv3x3_fwd(ALIGNED, ALIGNED, None, ALIGNED, *a, 0, None) == 1
    assert lib.conv3x3_dgrad(ALIGNED, ALIGNED, ALIGNED, *a, None) == 1
    assert lib.conv3x3_wgrad(ALIGNED, ALIGNED, ALIGNED, None, *a, ALIGNED, 1 << 30, None) == 1
    assert lib.conv3x3_wgrad_workspace_bytes(*a) == 0


def test_bad_pointers_and_enums_are_rejected_without_a_gpu(lib):
    a = (2, 64, 64, 8, 8)
    assert lib.conv3x3_fwd(None, ALIGNED, None, ALIGNED, *a, 0, None) == 1
    assert lib.conv3x3_fwd(ALIGNED + 2, ALIGNED, None, ALIGNED, *a, 0, None) == 1  # misaligned
    assert lib.conv3x3_fwd(ALIGNED, ALIGNED, None, ALIGNED, *a, 7, None) == 1      # bad act
    assert lib.conv3x3_fwd(ALIGNED, ALIGNED, None, ALIGNED, *a, 3, None) == 1      # one past LRELU
    assert lib.conv3x3_fwd(ALIGNED, ALIGNED, None, ALIGNED, *a, -1, None) == 1     # negative act
    assert lib.conv3x3_fwd_ex(ALIGNED, ALIGNED, None, ALIGNED, *a, 0, 5, 0, None) == 1  # dtype
    assert lib.conv3x3_fwd_ex(ALIGNED, ALIGNED, None, ALIGNED, *a, 0, 0, 9, None) == 1  # path
    assert lib.conv3x3_dgrad(ALIGNED, None, ALIGNED, *a, None) == 1
    assert lib.conv3x3_wgrad(ALIGNED, ALIGNED, None, None, *a, ALIGNED, 1 << 30, None) == 1
    # workspace that is required but missing / too small / misaligned
    need = lib.conv3x3_wgrad_workspace_bytes(*a)
    assert need > 0
    assert lib.conv3x3_wgrad(ALIGNED, ALIGNED, ALIGNED, None, *a, None, 0, None) == 5
    assert lib.conv3x3_wgrad(ALIGNED, ALIGNED, ALIGNED, None, *a, ALIGNED, need - 4, None) == 5
    assert lib.conv3x3_wgrad(ALIGNED, ALIGNED, ALIGNED, None, *a, ALIGNED + 16, need, None) == 1
    assert lib.conv3x3_fwd_f32(None, ALIGNED, None, ALIGNED, *a, 0, None) == 1


def test_fused_activation_entry_points_validate_without_a_gpu(lib):
    N, Cin, Cout, H, W = a = (2, 64, 64, 8, 8)
    far = ALIGNED + (1 << 24)            # a second fake buffer that overlaps nothing
    zb = N * H * W * Cout * 2            # bytes of z (bf16)
    # forward that also stores z: z missing, misaligned, overlapping y (either side)
    assert lib.conv3x3_fwd_save_z(ALIGNED, ALIGNED, None, far, None, *a, 1, 0, 0, None) == 1
    assert lib.conv3x3_fwd_save_z(ALIGNED, ALIGNED, None, far, far + (1 << 22) + 8, *a, 1, 0, 0,
                                  None) == 1
    assert lib.conv3x3_fwd_save_z(ALIGNED, ALIGNED, None, far, far + zb - 16, *a, 1, 0, 0,
                                  None) == 1
    assert lib.conv3x3_fwd_save_z(ALIGNED, ALIGNED, None, far + 4096, far, *a, 1, 0, 0, None) == 1
    # fp32 y is twice as long: z placed right after a bf16-sized y still overlaps it
    assert lib.conv3x3_fwd_save_z(ALIGNED, ALIGNED, None, far, far + zb, *a, 1, 1, 0, None) == 1
    # dgrad through an activation: unknown act_in, z_in missing / misaligned / overlapping dx
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, far, 3, ALIGNED, *a, 0, 0, None) == 1
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, far, -1, ALIGNED, *a, 0, 0, None) == 1
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, None, 1, ALIGNED, *a, 0, 0, None) == 1
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, far + 8, 2, ALIGNED, *a, 0, 0, None) == 1
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, far, 1, far + 256, *a, 0, 0, None) == 1
    # bad shape and bad dgrad arguments still come back as invalid
    assert lib.conv3x3_dgrad_act(ALIGNED, ALIGNED, far, 1, ALIGNED, 2, 60, 64, 8, 8, 0, 0,
                                 None) == 1
    assert lib.conv3x3_dgrad_act(None, ALIGNED, None, 0, ALIGNED, *a, 0, 0, None) == 1


def test_concat_free_entry_points_validate_without_a_gpu(lib):
    N, Cin, Cout, H, W = 2, 128, 64, 8, 8
    far = ALIGNED + (1 << 24)
    sh = (N, Cin, Cout, H, W)
    # bad split points, missing or misaligned second part
    for ca in (0, Cin, -8, 12):
        assert lib.conv3x3_fwd_cat(ALIGNED, far, ca, ALIGNED, None, ALIGNED, None, *sh, 1, 0, 0,
                                   None) == 1, ca
        assert lib.conv3x3_wgrad_cat(ALIGNED, far, ca, ALIGNED, ALIGNED, None, *sh, ALIGNED,
                                     1 << 30, 0, None) == 1, ca
        assert lib.conv3x3_wgrad_cat_workspace_bytes(N, Cin, ca, Cout, H, W, 0) == 0, ca
    assert lib.conv3x3_fwd_cat(ALIGNED, None, 64, ALIGNED, None, ALIGNED, None, *sh, 1, 0, 0,
                               None) == 1
    assert lib.conv3x3_fwd_cat(ALIGNED, far + 8, 64, ALIGNED, None, ALIGNED, None, *sh, 1, 0, 0,
                               None) == 1
    # z overlapping y
    assert lib.conv3x3_fwd_cat(ALIGNED, far, 64, ALIGNED, None, far + 4096, far + 4096 + 16, *sh,
                               1, 0, 0, None) == 1
    # dgrad: the two output parts overlap; z parts missing with an activation
    assert lib.conv3x3_dgrad_cat(ALIGNED, ALIGNED, far, far + 64, 64, None, None, 0, *sh, 0, 0,
                                 None) == 1
    assert lib.conv3x3_dgrad_cat(ALIGNED, ALIGNED, far, far + (1 << 22), 64, None, None, 1, *sh, 0,
                                 0, None) == 1
    assert lib.conv3x3_dgrad_cat(ALIGNED, ALIGNED, far, far + (1 << 22), 64, ALIGNED, ALIGNED, 5,
                                 *sh, 0, 0, None) == 1
    # a split that is not a whole 64-channel chunk cannot be forced onto the tensor cores
    assert lib.conv3x3_wgrad_cat_workspace_bytes(N, Cin, 32, Cout, H, W, 1) == 0
    assert lib.conv3x3_wgrad_cat_workspace_bytes(N, Cin, 32, Cout, H, W, 0) > 0
    # a tensor-core split needs the same scratch as the unsplit call
    assert (lib.conv3x3_wgrad_cat_workspace_bytes(N, Cin, 64, Cout, H, W, 0)
            == lib.conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W))


def test_strided_entry_points_validate_without_a_gpu(lib):
    sh = (2, 64, 64, 8, 8)
    far = ALIGNED + (1 << 24)
    for bad in (0, 3, -1):
        assert lib.conv3x3_fwd_strided(ALIGNED, ALIGNED, None, far, None, *sh, bad, 0, 0, 0,
                                       None) == 1, bad
        assert lib.conv3x3_dgrad_strided(ALIGNED, ALIGNED, far, None, 0, *sh, bad, 0, 0,
                                         None) == 1, bad
        assert lib.conv3x3_wgrad_strided(ALIGNED, ALIGNED, ALIGNED, None, *sh, bad, ALIGNED,
                                         1 << 30, 0, None) == 1, bad
        assert lib.conv3x3_wgrad_strided_workspace_bytes(*sh, bad, 0) == 0
    # z overlapping y (y is [2][4][4][64] bf16 = 4 KB); z_in missing with an activation
    assert lib.conv3x3_fwd_strided(ALIGNED, ALIGNED, None, far, far + 2048, *sh, 2, 1, 0, 0,
                                   None) == 1
    assert lib.conv3x3_dgrad_strided(ALIGNED, ALIGNED, far, None, 1, *sh, 2, 0, 0, None) == 1
    # stride 2 on the tensor cores needs 64 channels each side; the split plan runs over dy's grid
    assert lib.conv3x3_wgrad_strided_workspace_bytes(2, 32, 64, 8, 8, 2, 1) == 0
    assert lib.conv3x3_wgrad_strided_workspace_bytes(2, 32, 64, 8, 8, 2, 0) > 0
    assert (lib.conv3x3_wgrad_strided_workspace_bytes(64, 128, 128, 64, 64, 2, 0)
            == lib.conv3x3_wgrad_workspace_bytes(64, 128, 128, 32, 32))
    assert (lib.conv3x3_wgrad_strided_workspace_bytes(*sh, 1, 0)
            == lib.conv3x3_wgrad_workspace_bytes(*sh))


def test_workspace_size_depends_only_on_shape(lib):
    from synth import STACK, STEM, L1, L2, L3
    for L in [STEM, L1, L2, L3] + STACK:
        a = (L.N, L.Cin, L.Cout, L.H, L.W)
        n = lib.conv3x3_wgrad_workspace_bytes(*a)
        assert n == lib.conv3x3_wgrad_workspace_bytes(*a)
        assert n >= 4 * (L.Cout * 9 * L.Cin + L.Cout)  # at least one full partial slice
        assert n < 1 << 31


def test_auto_path_is_host_only_and_valid(lib):
    assert lib.conv3x3_auto_path(0, 64, 128, 128, 64, 64) in (1, 2)
    assert lib.conv3x3_auto_path(0, 64, 3, 128, 64, 64) == -1
