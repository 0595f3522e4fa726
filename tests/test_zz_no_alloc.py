"""conv3x3_wgrad_noalloc: the weight gradient for callers that cannot allocate
device memory (a plugin whose host application owns the memory pool, or a
latency-critical loop that may not call cudaMalloc after start-up).  Its
split-K scratch is a fixed array inside the library, so these tests check it
against conv3x3_wgrad with caller-provided scratch, twice in a row (the second
call reuses whatever the first left in the shared array).

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
from x3_convolution_gb300 import _lib as L
from x3_convolution_gb300 import ops

from gpu_util import rel_err, to_dev_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the gate the other wgrad parity tests use for fp32 dw / db


def _inputs(shape, seed):
    N, Cin, Cout, H, W = shape
    t = synth.make_tensors(synth.Layer("na", N, Cin, Cout, H, W), seed=seed)
    return to_dev_bf16(t.x), to_dev_bf16(t.dy)


@pytest.mark.parametrize("shape", [(2, 64, 128, 8, 8), (64, 128, 128, 64, 64), (3, 72, 200, 9, 11)],
                         ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_wgrad_on_two_calls_in_a_row(shape):
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    N, Cin, Cout, H, W = shape
    assert L.conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W) <= L.WGRAD_NOALLOC_MAX_BYTES
    x, dy = _inputs(shape, seed=11)
    ref_dw, ref_db = ops.wgrad(x, dy)
    outs = []
    for _ in range(2):
        dw = torch.full((Cout, 3, 3, Cin), float("nan"), device="cuda")
        db = torch.full((Cout,), float("nan"), device="cuda")
        L.conv3x3_wgrad_noalloc(x, dy, dw, db, N, Cin, Cout, H, W)
        outs.append((dw, db))
    torch.cuda.synchronize()
    assert L.conv3x3_device_status() == L.OK
    r_dw = ref_dw.double().cpu().numpy()
    r_db = ref_db.double().cpu().numpy()
    for dw, db in outs:
        assert rel_err(dw.double().cpu().numpy(), r_dw) <= TOL
        assert rel_err(db.double().cpu().numpy(), r_db) <= TOL


def test_noalloc_after_a_different_shape():
    # a larger call leaves more of the shared array written than a smaller one reads
    for shape in [(8, 256, 256, 16, 16), (2, 64, 64, 8, 8)]:
        N, Cin, Cout, H, W = shape
        x, dy = _inputs(shape, seed=5)
        ref_dw, ref_db = ops.wgrad(x, dy)
        dw = torch.empty((Cout, 3, 3, Cin), device="cuda")
        db = torch.empty((Cout,), device="cuda")
        L.conv3x3_wgrad_noalloc(x, dy, dw, db, N, Cin, Cout, H, W)
        torch.cuda.synchronize()
        assert rel_err(dw.double().cpu().numpy(), ref_dw.double().cpu().numpy()) <= TOL
        assert rel_err(db.double().cpu().numpy(), ref_db.double().cpu().numpy()) <= TOL


def test_noalloc_allocates_no_device_memory():
    # after a first call (which loads the kernels and looks up the array), a
    # call leaves the device's free memory exactly where it was
    N, Cin, Cout, H, W = 16, 128, 128, 32, 32
    x, dy = _inputs((N, Cin, Cout, H, W), seed=3)
    dw = torch.empty((Cout, 3, 3, Cin), device="cuda")
    db = torch.empty((Cout,), device="cuda")
    L.conv3x3_wgrad_noalloc(x, dy, dw, db, N, Cin, Cout, H, W)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        L.conv3x3_wgrad_noalloc(x, dy, dw, db, N, Cin, Cout, H, W)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert L.conv3x3_device_status() == L.OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 2048 -> 2048 channels: one dw partial alone is ~151 MB
    N, Cin, Cout, H, W = 64, 2048, 2048, 8, 8
    assert L.conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W) > L.WGRAD_NOALLOC_MAX_BYTES
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.Conv3x3Error) as e:
        L.conv3x3_wgrad_noalloc(dummy, dummy, dummy, None, N, Cin, Cout, H, W)
    assert e.value.status == L.ERR_WORKSPACE
