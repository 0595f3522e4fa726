#!/usr/bin/env python3
"""Benchmark: 3x3 conv fwd + dgrad + wgrad throughput (TFLOP/s) on GB300.

One step = one training-step sweep over the UNet's 3x3 convs: every layer's
forward (bias + SiLU epilogue) in network order, then every dgrad in reverse
order, then every wgrad (+ dbias) in reverse order, each through the C ABI of
libconv3x3.so on one stream.  CUDA events at the step's start and at the end of
each pass give the step time and the per-pass times.

Default workload "unet": the stem conv (3 -> 128 channels, zero-padded to 8,
64x64) followed by the 32 resblock convs of the 64x64 diffusion UNet (base 128,
multipliers 1,2,3,4, two resblocks per level on the down and up paths, up-path
inputs = concat of skip and main), batch 64, bf16 NHWC, seeded synthetic inputs.

--concat-free gives each up-path conv its main branch and its skip as two
tensors (conv3x3_fwd_cat / conv3x3_dgrad_cat / conv3x3_wgrad_cat): no
concatenated input is built and dx comes back already split.

--fused-act runs the training step with the activation's backward fused into
the convolutions: each forward also stores its pre-activation z
(conv3x3_fwd_save_z) and each dgrad takes the pre-activation of the layer that
produced its input and returns the gradient through that activation
(conv3x3_dgrad_act), so no elementwise pass runs between the convolutions.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream; L2 is flushed between steps, outside the events: a write of
a buffer twice the L2 size, then a read of a second such buffer, so that the
dirty lines the write leaves are written back before the timed region starts
(the timed kernels find L2 cold and clean).  Multi-process runs (torchrun) run one replica per GPU
(weak scaling); the reported time is the max over ranks.

Beside the step, the line carries the per-layer breakdown of the step
(layers_detail: extra untimed steps with an event pair around every call) and
the gates block: each pass of the per-layer workloads (stem, l1, l2, l3) timed
alone with L2 flushed before every call, as a fraction of its roofline (HBM for
the 8-input-channel stem, the dense bf16 tensor peak for the others) against
its target, and the tiny fp32 check workload (launch-bound, no target).

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload: each step runs fwd + dgrad + wgrad of one image of
one layer, cycling through the layers.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "3x3 conv fwd+dgrad+wgrad TFLOP/s on 1 GB300 and % of roofline"
UNIT = "TFLOP/s"


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------
def layer_bytes(L: synth.Layer):
    """Algorithmic HBM bytes per pass: each ABI tensor read or written once."""
    x = L.P * L.Cin * 2
    dy = L.Po * L.Cout * 2                  # y and dy live on the output grid
    w = L.Cout * 9 * L.Cin * 2
    fwd = x + w + dy + L.Cout * 4           # x, w, bias in; y out
    dgrad = dy + w + x                      # dy, w in; dx out
    wgrad = x + dy + L.Cout * 9 * L.Cin * 4 + L.Cout * 4  # x, dy in; dw, db out
    return {"fwd": fwd, "dgrad": dgrad, "wgrad": wgrad}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def roofline_time_s(L, peaks, tflops_key="bf16_tflops"):
    by = layer_bytes(L)
    f = L.flops_per_pass()
    return {k: max(f / (peaks[tflops_key] * 1e12), by[k] / (peaks["hbm_gbs"] * 1e9)) for k in by}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
def gpu_selector(device) -> str:
    """nvidia-smi -i argument for a torch device (its UUID when torch exposes it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    idx = device.index or 0
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    return ids[idx] if idx < len(ids) else str(idx)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def whole_job_tflops(flops_per_rank_step: float, ws: int, ms_max: float) -> float:
    """Weak scaling: every rank runs the same step; the job's throughput is all ranks'
    FLOPs over the slowest rank's time."""
    return flops_per_rank_step * ws / (ms_max * 1e-3) / 1e12


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
class Workload:
    def __init__(self, layers, seed, device, keep_host=True, fused_act=False, concat_free=False,
                 path=0):
        import torch
        self.layers = layers
        self.fused_act = fused_act
        self.concat_free = concat_free
        self.path = path  # kernel family of the plain calls (0 = AUTO)
        self.dev = []
        self.host = []
        ws_max = 0
        from x3_convolution_gb300 import _lib as Lb
        for i, L in enumerate(layers):
            t = synth.make_tensors(L, seed=seed, index=i)
            hx = torch.from_numpy(synth.bf16_bits(t.x).view(np.int16)).view(torch.bfloat16)
            hw = torch.from_numpy(synth.bf16_bits(t.w).view(np.int16)).view(torch.bfloat16)
            hb = torch.from_numpy(t.bias.copy())
            hdy = torch.from_numpy(synth.bf16_bits(t.dy).view(np.int16)).view(torch.bfloat16)
            del t
            d = {
                "x": hx.to(device), "w": hw.to(device), "b": hb.to(device), "dy": hdy.to(device),
                "y": torch.empty((L.N, L.Ho, L.Wo, L.Cout), dtype=torch.bfloat16, device=device),
                "dx": torch.empty((L.N, L.H, L.W, L.Cin), dtype=torch.bfloat16, device=device),
                "dw": torch.empty((L.Cout, 3, 3, L.Cin), dtype=torch.float32, device=device),
                "db": torch.empty((L.Cout,), dtype=torch.float32, device=device),
            }
            cat = concat_free and L.cat_a > 0
            d["cat_a"] = L.cat_a if cat else 0
            if cat:
                # up-path conv: main and skip stay two tensors; no concat buffer
                ca = L.cat_a
                d["xa"] = d["x"][..., :ca].contiguous()
                d["xb"] = d["x"][..., ca:].contiguous()
                d["dxa"] = torch.empty((L.N, L.H, L.W, ca), dtype=torch.bfloat16, device=device)
                d["dxb"] = torch.empty((L.N, L.H, L.W, L.Cin - ca), dtype=torch.bfloat16,
                                       device=device)
                del d["x"], d["dx"]
            if fused_act:
                # z: this layer's pre-activation (written by the forward);
                # zin: the pre-activation of the layer that produced x (none for
                # the stem, whose input is the image)
                d["z"] = torch.empty((L.N, L.Ho, L.Wo, L.Cout), dtype=torch.bfloat16, device=device)
                d["act_in"] = L.act if i > 0 else 0
                hz = torch.from_numpy(synth.bf16_bits(synth.make_zin(L, seed=seed, index=i))
                                      .view(np.int16)).view(torch.bfloat16)
                d["zin"] = hz.to(device)
                if cat:
                    d["za"] = d["zin"][..., :L.cat_a].contiguous()
                    d["zb"] = d["zin"][..., L.cat_a:].contiguous()
                    del d["zin"]
            self.dev.append(d)
            if keep_host:
                h = {"x": hx.pin_memory(), "w": hw.pin_memory(), "b": hb.pin_memory(),
                     "dy": hdy.pin_memory(),
                     "dw": torch.empty((L.Cout, 3, 3, L.Cin), dtype=torch.float32).pin_memory(),
                     "db": torch.empty((L.Cout,), dtype=torch.float32).pin_memory()}
                if fused_act:
                    h["zin"] = hz.pin_memory()
                if cat:
                    ca = L.cat_a
                    h["xa"] = h["x"][..., :ca].contiguous().pin_memory()
                    h["xb"] = h["x"][..., ca:].contiguous().pin_memory()
                    del h["x"]
                    if fused_act:
                        h["za"] = h["zin"][..., :ca].contiguous().pin_memory()
                        h["zb"] = h["zin"][..., ca:].contiguous().pin_memory()
                        del h["zin"]
                self.host.append(h)
            if L.stride != 1:
                ws_max = max(ws_max, Lb.conv3x3_wgrad_strided_workspace_bytes(
                    L.N, L.Cin, L.Cout, L.H, L.W, L.stride, Lb.PATH_AUTO))
            elif cat:
                ws_max = max(ws_max, Lb.conv3x3_wgrad_cat_workspace_bytes(
                    L.N, L.Cin, L.cat_a, L.Cout, L.H, L.W, Lb.PATH_AUTO))
            else:
                ws_max = max(ws_max, Lb.conv3x3_wgrad_workspace_bytes_ex(L.N, L.Cin, L.Cout, L.H, L.W,
                                                                         path))
        self.ws_bytes = ws_max
        self.ws = torch.empty(max(ws_max, 256), dtype=torch.uint8, device=device)
        # one more split-K workspace per extra wgrad stream (see run_step)
        self.ws_side = []
        self.device = device

    def side_workspace(self, k):
        import torch
        while len(self.ws_side) <= k:
            self.ws_side.append(torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8,
                                            device=self.device))
        return self.ws_side[k]

    def inputs(self, h):
        keys = ("x", "xa", "xb", "w", "b", "dy", "zin", "za", "zb")
        return [k for k in keys if k in h]

    def h2d_bytes(self):
        return sum(h[k].numel() * h[k].element_size() for h in self.host for k in self.inputs(h))

    def d2h_bytes(self):
        return sum(h[k].numel() * h[k].element_size() for h in self.host for k in ("dw", "db"))


def _fwd(wl, i, sh):
    from x3_convolution_gb300 import _lib as Lb
    L, d = wl.layers[i], wl.dev[i]
    if L.stride != 1:
        Lb.conv3x3_fwd_strided(d["x"], d["w"], d["b"], d["y"], d.get("z"), L.N, L.Cin, L.Cout, L.H,
                               L.W, L.stride, L.act, Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif d["cat_a"]:
        Lb.conv3x3_fwd_cat(d["xa"], d["xb"], d["cat_a"], d["w"], d["b"], d["y"], d.get("z"), L.N,
                           L.Cin, L.Cout, L.H, L.W, L.act, Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif wl.fused_act:
        Lb.conv3x3_fwd_save_z(d["x"], d["w"], d["b"], d["y"], d["z"], L.N, L.Cin, L.Cout, L.H, L.W,
                              L.act, Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif getattr(wl, "path", 0):
        Lb.conv3x3_fwd_ex(d["x"], d["w"], d["b"], d["y"], L.N, L.Cin, L.Cout, L.H, L.W, L.act,
                          Lb.DT_BF16, wl.path, sh)
    else:
        Lb.conv3x3_fwd(d["x"], d["w"], d["b"], d["y"], L.N, L.Cin, L.Cout, L.H, L.W, L.act, sh)
    return 1


def _dgrad(wl, i, sh):
    from x3_convolution_gb300 import _lib as Lb
    L, d = wl.layers[i], wl.dev[i]
    if L.stride != 1:
        Lb.conv3x3_dgrad_strided(d["dy"], d["w"], d["dx"], d.get("zin"), d.get("act_in", 0), L.N,
                                 L.Cin, L.Cout, L.H, L.W, L.stride, Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif d["cat_a"]:
        Lb.conv3x3_dgrad_cat(d["dy"], d["w"], d["dxa"], d["dxb"], d["cat_a"], d.get("za"),
                             d.get("zb"), d.get("act_in", 0), L.N, L.Cin, L.Cout, L.H, L.W,
                             Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif wl.fused_act:
        Lb.conv3x3_dgrad_act(d["dy"], d["w"], d["zin"], d["act_in"], d["dx"], L.N, L.Cin, L.Cout,
                             L.H, L.W, Lb.DT_BF16, Lb.PATH_AUTO, sh)
    elif getattr(wl, "path", 0):
        Lb.conv3x3_dgrad_ex(d["dy"], d["w"], d["dx"], L.N, L.Cin, L.Cout, L.H, L.W, Lb.DT_BF16,
                            wl.path, sh)
    else:
        Lb.conv3x3_dgrad(d["dy"], d["w"], d["dx"], L.N, L.Cin, L.Cout, L.H, L.W, sh)
    return 1


def _wgrad(wl, i, sh, side=-1):
    from x3_convolution_gb300 import _lib as Lb
    L, d = wl.layers[i], wl.dev[i]
    ws = wl.side_workspace(side) if side >= 0 else wl.ws
    if L.stride != 1:
        Lb.conv3x3_wgrad_strided(d["x"], d["dy"], d["dw"], d["db"], L.N, L.Cin, L.Cout, L.H, L.W,
                                 L.stride, ws, wl.ws_bytes, Lb.PATH_AUTO, sh)
    elif d["cat_a"]:
        Lb.conv3x3_wgrad_cat(d["xa"], d["xb"], d["cat_a"], d["dy"], d["dw"], d["db"], L.N, L.Cin,
                             L.Cout, L.H, L.W, ws, wl.ws_bytes, Lb.PATH_AUTO, sh)
    elif getattr(wl, "path", 0):
        Lb.conv3x3_wgrad_ex(d["x"], d["dy"], d["dw"], d["db"], L.N, L.Cin, L.Cout, L.H, L.W, ws,
                            wl.ws_bytes, wl.path, sh)
    else:
        Lb.conv3x3_wgrad(d["x"], d["dy"], d["dw"], d["db"], L.N, L.Cin, L.Cout, L.H, L.W, ws,
                         wl.ws_bytes, sh)
    return 2  # partial-sum kernel + fixed-order reduction


# DRAM bytes per call (dram__bytes_read.sum + dram__bytes_write.sum) of each
# pass on the per-layer configs (stem, l1, l2, l3), from one scoped ncu capture
# per config -- every launch of the call (the weight gradient's kernel and its
# reduction), DRAM counters only, one pass each, caches flushed by ncu before
# each launch, so the reduction reads its split-K partials from DRAM here where
# in a step they are still in L2, and writes still in L2 when a kernel ends are
# not counted -- and the SHA-256 of the kernel sources they were taken on: a
# figure is reported only while those sources are unchanged.  Command: for each
# config, ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,
# gpu__time_duration.sum --clock-control none -k regex:"k_(igemm|wgrad|stem)"
# -s 12 -c 4 on bench.py --workload <config> --steps 1 --warmup 3 --no-e2e
# --no-cpu-baseline --no-detail --no-gates --no-graph --wgrad-streams 1.
RECORDED_TRAFFIC: dict = {   # {(config, pass): bytes per call}
    ("stem", "fwd"): 11126528, ("stem", "dgrad"): 67164928, ("stem", "wgrad"): 77080576,
    ("l1", "fwd"): 91249408, ("l1", "dgrad"): 87177216, ("l1", "wgrad"): 165513984,
    ("l2", "fwd"): 34787072, ("l2", "dgrad"): 34812672, ("l2", "wgrad"): 95642624,
    ("l3", "fwd"): 15273216, ("l3", "dgrad"): 15263232, ("l3", "wgrad"): 51759360,
}
# DRAM bytes of each pass of the UNet step (the pass's launches summed: 33
# forwards, 33 input gradients, 33 weight gradients with their reductions),
# from one scoped capture of a whole step's 133 launches -- one pass per
# launch, caches flushed by ncu before each, writes still in L2 at a launch's
# end not counted -- valid under the same source hash.  Command: ncu --metrics
# dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
# --clock-control none -k regex:"k_(igemm|wgrad|stem)" -s 399 -c 133 on
# bench.py --steps 1 --warmup 3 --no-e2e --no-cpu-baseline --no-detail
# --no-gates --no-graph --wgrad-streams 1.
RECORDED_STEP_TRAFFIC: dict = {"fwd": 1544771584, "dgrad": 1463119872, "wgrad": 3211335680}
TRAFFIC_SOURCES = ("tc.cu", "simt.cu", "ptx.cuh", "conv3x3_internal.h")
TRAFFIC_SHA256 = "68892b132c3be8c4bbd9cb2a5ba20b5380147d74b1cb70940856ed614dd8cc75"


# The six resampling ops of a step, the same way: ncu --metrics (as above)
# -k regex:"k_upfirdn2d" -s 18 -c 6 on bench.py --workload upfirdn2d --steps 1
# --warmup 3 --no-e2e --no-cpu-baseline.
RECORDED_UFD_TRAFFIC = 235442176
UFD_SOURCES = ("upfirdn2d.cu", "conv3x3_internal.h")
UFD_SHA256 = "76b05b309ae5258121dd03bff3684fb85d605294f6da4de386dce5e1a5991dc1"


def sources_sha256(files=None):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "x3_convolution_gb300", "csrc")
    try:
        for f in (files or TRAFFIC_SOURCES):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return h.hexdigest()


def recorded_traffic(config, pas):
    """Bytes per call of `pas` on per-layer config `config` from the recorded
    capture, or None when there is none or the kernels changed since."""
    if TRAFFIC_SHA256 is None or (config, pas) not in RECORDED_TRAFFIC:
        return None
    return RECORDED_TRAFFIC[(config, pas)] if sources_sha256() == TRAFFIC_SHA256 else None


def recorded_pass_traffic(workload, pas, fused_act=False, concat_free=False, path="auto"):
    """DRAM bytes per step of pass `pas` for the bench line's roofline: the
    recorded whole-step capture for the UNet step, the per-call capture for a
    per-layer config; None for any other workload or variant (the fused or
    concat-free calls and forced paths run other kernels than those captured)
    and when the kernels changed since."""
    if fused_act or concat_free or path != "auto" or TRAFFIC_SHA256 is None:
        return None
    if workload == "unet":
        t = RECORDED_STEP_TRAFFIC.get(pas)
        return t if t is not None and sources_sha256() == TRAFFIC_SHA256 else None
    return recorded_traffic(workload, pas)


def pick_peak(peaks, clocks, timed_s):
    """The tensor peak the step is held to: the burst figure (cuBLAS timed in
    isolation) when the timed region is short and the SM clock stayed near its
    maximum, else the sustained one (cuBLAS held for seconds under the power cap)."""
    burst = clocks is not None and timed_s < 1.0 and \
        clocks.get("sm_mhz", 0.0) >= 0.95 * clocks.get("sm_max_mhz", 1e9)
    key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    return key, peaks[key]


# The per-layer workloads and the gate each is held to: the small-channel stem
# against the HBM roofline, the large-channel layers against the dense bf16
# tensor peak (burst: each call is timed alone).
GATES = (("stem", "hbm", 0.70), ("l1", "tensor", 0.60), ("l2", "tensor", 0.60),
         ("l3", "tensor", 0.60))


class L2Flush:
    """Evicts L2 on the current stream: writes a buffer twice the L2 size, then
    reads a second one, so that the write's dirty lines reach DRAM here and not
    inside the next timed region."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 64 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)
        self.bytes = 2 * 4 * n

    def __call__(self):
        self.w.zero_()
        self.r.sum()


FLUSH_NOTE = "flushed between steps (write of 2x L2, then a read of another 2x L2)"


def call_us(stream, flush, fn, warm=3, reps=15):
    """Median device time of fn() (one C ABI call) in microseconds: CUDA events
    on the launching stream around the call only, L2 flushed before each run."""
    import torch
    evs = []
    for r in range(warm + reps):
        with torch.cuda.stream(stream):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
        if r >= warm:
            evs.append((a, b))
    stream.synchronize()
    return float(np.median([a.elapsed_time(b) * 1e3 for a, b in evs]))


def config_gates(seed, device, stream, flush, peaks):
    """Each pass of each per-layer workload timed alone, as a fraction of its
    roofline, against its target; and the tiny fp32 check workload (launch-bound,
    no target)."""
    import torch
    from x3_convolution_gb300 import _lib as Lb
    sh = stream.cuda_stream
    out = {}
    for name, bound, target in GATES:
        L = synth.CONFIGS[name][0]
        wl = Workload([L], seed, device, keep_host=False)
        rt = roofline_time_s(L, peaks)
        rs = roofline_time_s(L, peaks, "bf16_tflops_sustained")
        by = layer_bytes(L)
        ent = {"bound": bound, "target": target, "shape": [L.N, L.Cin, L.Cout, L.H, L.W]}
        for k, fn in (("fwd", _fwd), ("dgrad", _dgrad), ("wgrad", _wgrad)):
            us = call_us(stream, flush, lambda: fn(wl, 0, sh))
            frac = rt[k] / (us * 1e-6)
            e = {"us": round(us, 2), "tflops": round(L.flops_per_pass() / (us * 1e-6) / 1e12, 1),
                 "gbs": round(by[k] / (us * 1e-6) / 1e9, 1), "frac": round(frac, 3),
                 "pass": bool(frac >= target), "traffic": recorded_traffic(name, k),
                 "algorithmic_bytes": by[k]}
            if bound == "tensor":
                e["frac_sustained"] = round(rs[k] / (us * 1e-6), 3)
            ent[k] = e
        out[name] = ent
        del wl
        torch.cuda.empty_cache()
    # tiny: the fp32 check path (CUDA-core fp32 FMA); launch-bound, parity only
    T = synth.TINY
    t = synth.make_tensors(T, seed=seed)
    x, w, b, dy = (torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
                   for a in (t.x, t.w, t.bias, t.dy))
    y = torch.empty((T.N, T.H, T.W, T.Cout), dtype=torch.float32, device=device)
    dx = torch.empty_like(x)
    dw = torch.empty((T.Cout, 3, 3, T.Cin), dtype=torch.float32, device=device)
    db = torch.empty((T.Cout,), dtype=torch.float32, device=device)
    tiny = {"bound": "launch", "target": None, "shape": [T.N, T.Cin, T.Cout, T.H, T.W],
            "dtype": "f32"}
    for k, fn in (("fwd", lambda: Lb.conv3x3_fwd_f32(x, w, b, y, T.N, T.Cin, T.Cout, T.H, T.W, 0, sh)),
                  ("dgrad", lambda: Lb.conv3x3_dgrad_f32(dy, w, dx, T.N, T.Cin, T.Cout, T.H, T.W, sh)),
                  ("wgrad", lambda: Lb.conv3x3_wgrad_f32(x, dy, dw, db, T.N, T.Cin, T.Cout, T.H,
                                                        T.W, None, 0, sh))):
        tiny[k] = {"us": round(call_us(stream, flush, fn), 2)}
    out["tiny"] = tiny
    return out


def run_step(wl: Workload, stream_handle: int, record=None, mark=None, interleave=False,
             streams=None):
    """One sweep through the C ABI: every layer's forward in network order, then
    the backward in reverse order -- by default every dgrad, then every wgrad (a
    wgrad needs only its layer's x and dy); with `interleave` each layer's
    dgrad and wgrad back to back.  `record(kind, i, 0|1)` brackets each call,
    `mark(pass)` the end of each pass.  With `streams` = (main, side, ...) torch
    streams (main being the stream of `stream_handle`), the wgrad calls -- which
    depend on no other wgrad -- go round-robin over the streams (fork and join
    by events, each stream with its own workspace), so that one layer's
    reduction and last tile round overlap the next layer's wgrad.  The forward
    and dgrad calls stay in order on one stream: in a network each depends on
    the one before.  Returns the number of kernel launches."""
    def call(kind, fn, i):
        if record is not None:
            record(kind, i, 0)
        k = fn(wl, i, stream_handle)
        if record is not None:
            record(kind, i, 1)
        return k

    n = 0
    if mark is not None:
        mark("start")
    for i in range(len(wl.layers)):
        n += call("fwd", _fwd, i)
    if mark is not None:
        mark("fwd")
    back = list(reversed(range(len(wl.layers))))
    if interleave:
        for i in back:
            n += call("dgrad", _dgrad, i)
            n += call("wgrad", _wgrad, i)
        return n
    for i in back:
        n += call("dgrad", _dgrad, i)
    if mark is not None:
        mark("dgrad")
    if streams is None:
        for i in back:
            n += call("wgrad", _wgrad, i)
    else:
        import torch
        main, sides = streams[0], streams[1:]
        for sd in sides:
            sd.wait_stream(main)
        for j, i in enumerate(back):
            k = j % len(streams)
            if k:
                n += _wgrad(wl, i, sides[k - 1].cuda_stream, side=k - 1)
            else:
                n += call("wgrad", _wgrad, i)
        for sd in sides:
            main.wait_stream(sd)
    if mark is not None:
        mark("wgrad")
    return n


def cuda_arm(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    import __graft_entry__ as ge
    ge.build()
    from x3_convolution_gb300 import _lib as Lb

    layers = synth.CONFIGS[args.workload]
    peaks = load_peaks()
    path = {"auto": Lb.PATH_AUTO, "tensor": Lb.PATH_TENSOR, "simt": Lb.PATH_SIMT}[args.path]
    wl = Workload(layers, args.seed, device, keep_host=not args.no_e2e, fused_act=args.fused_act,
                  concat_free=args.concat_free, path=path)
    stream = torch.cuda.Stream(device=device)
    sh = stream.cuda_stream
    # the wgrad pass runs on --wgrad-streams streams (1: in order on one)
    wstreams = None
    if args.wgrad_streams > 1:
        wstreams = (stream,) + tuple(torch.cuda.Stream(device=device)
                                     for _ in range(args.wgrad_streams - 1))
    flush = L2Flush(device)

    flops_step = sum(3 * L.flops_per_pass() for L in layers)
    flops_padded = sum(3 * L.flops_per_pass(padded=True) for L in layers)

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run_step(wl, sh, streams=wstreams)
    torch.cuda.synchronize(device)
    st = Lb.conv3x3_device_status(sh)
    if st != Lb.OK:
        raise RuntimeError("device status after warm-up: " + Lb.status_string(st))

    # Timed steps: CUDA events on the launching stream at the step's start and
    # at the end of each pass (forward, dgrad, wgrad).  By default the step's
    # C ABI calls and these events are captured once into a CUDA graph that
    # each timed step replays on the same stream (the launches of 132 kernels
    # then cost the GPU no gaps); --no-graph launches them one by one.
    # Per-call events (the per-layer detail) are recorded in extra steps after the timed
    # region.
    fam_ms = {"fwd": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    marks = {}

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        marks[name] = e

    def mark_in_graph(name):
        # an event record node of the graph (re-recorded at every replay)
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record(stream)
        marks[name] = e

    graph = None
    launches_per_step = 0
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            launches_per_step = run_step(wl, sh, mark=mark_in_graph, streams=wstreams)
        torch.cuda.synchronize(device)
        for _ in range(args.warmup):
            with torch.cuda.stream(stream):
                graph.replay()
        torch.cuda.synchronize(device)

    sampler = ClockSampler(gpu_selector(device))
    sampler.start()
    time.sleep(0.3)
    step_ms = []
    launches = 0
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            flush()  # same stream, before the start event: evict L2
            if graph is not None:
                graph.replay()
                launches += launches_per_step
        if graph is None:
            launches += run_step(wl, sh, mark=mark, streams=wstreams)
        torch.cuda.synchronize(device)
        step_ms.append(marks["start"].elapsed_time(marks["wgrad"]))
        fam_ms["fwd"] += marks["start"].elapsed_time(marks["fwd"])
        fam_ms["dgrad"] += marks["fwd"].elapsed_time(marks["dgrad"])
        fam_ms["wgrad"] += marks["dgrad"].elapsed_time(marks["wgrad"])
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    st = Lb.conv3x3_device_status(sh)
    if st != Lb.OK:
        raise RuntimeError("device status after timed steps: " + Lb.status_string(st))

    ms = float(np.mean(step_ms))
    ms_max = max_over_ranks(ms, ws, device)
    value = whole_job_tflops(flops_step, ws, ms_max)

    # per-pass breakdown and the roofline of the dominant kernel family
    K = args.steps
    fam = {}
    fl = sum(L.flops_per_pass() for L in layers)
    for k in ("fwd", "dgrad", "wgrad"):
        t = fam_ms[k] / K  # ms per step
        fam[k] = {"ms_per_step": round(float(t), 4), "tflops": round(fl / (t * 1e-3) / 1e12, 1)}
    dom = max(fam, key=lambda k: fam[k]["ms_per_step"])
    achieved = fl / (fam[dom]["ms_per_step"] * 1e-3) / 1e12
    peak_key, peak = pick_peak(peaks, clocks, sum(step_ms) * 1e-3)
    roof_s = sum(sum(roofline_time_s(L, peaks).values()) for L in layers)

    # per-layer detail: extra (untimed) steps with an event pair around every call
    per_layer = None
    if not args.no_detail:
        nlay = len(layers)
        per_call = {k: [[None, None] for _ in range(nlay)] for k in fam}
        call_ms = {k: np.zeros(nlay) for k in fam}

        def record(kind, i, which):
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            per_call[kind][i][which] = e

        nd = max(3, min(K, 10))
        for _ in range(nd):
            with torch.cuda.stream(stream):
                flush()
            run_step(wl, sh, record=record)
            torch.cuda.synchronize(device)
            for k in per_call:
                for i in range(nlay):
                    a, b = per_call[k][i]
                    call_ms[k][i] += a.elapsed_time(b)
        per_layer = []
        for i, L in enumerate(layers):
            rt = roofline_time_s(L, peaks)
            per_layer.append({
                "name": L.name, "N": L.N, "Cin": L.Cin, "Cout": L.Cout, "H": L.H, "W": L.W,
                "stride": L.stride,
                "path": {k: ["auto", "tensor", "simt"][max(0, Lb.conv3x3_auto_path(j, L.N, L.Cin, L.Cout, L.H, L.W))]
                         for j, k in enumerate(("fwd", "dgrad", "wgrad"))},
                "us": {k: round(float(call_ms[k][i] / nd * 1e3), 2) for k in call_ms},
                "tflops": {k: round(L.flops_per_pass() / (call_ms[k][i] / nd * 1e-3) / 1e12, 1) for k in call_ms},
                "roofline_frac": {k: round(rt[k] / (call_ms[k][i] / nd * 1e-3), 3) for k in call_ms},
            })

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        # Pipelined through the public calls: one stream uploads every layer's
        # forward inputs (network order) and then its dy (reverse order, the
        # order the backward consumes them); the compute stream waits only for
        # the layer it is about to run, and runs each layer's dgrad and wgrad
        # back to back so that the backward trails the uploads closely; a third
        # stream downloads each layer's dw and dbias as soon as its wgrad is done.
        up = torch.cuda.Stream(device=device)
        down = torch.cuda.Stream(device=device)
        nl = len(wl.layers)
        ev_fwd_in = [torch.cuda.Event() for _ in range(nl)]
        ev_dy_in = [torch.cuda.Event() for _ in range(nl)]
        ev_grads = [torch.cuda.Event() for _ in range(nl)]

        def hook(kind, i, which):
            if kind == "fwd" and which == 0:
                stream.wait_event(ev_fwd_in[i])
            elif kind == "dgrad" and which == 0:
                stream.wait_event(ev_dy_in[i])
            elif kind == "wgrad" and which == 1:
                ev_grads[i].record(stream)
                down.wait_event(ev_grads[i])
                with torch.cuda.stream(down):
                    wl.host[i]["dw"].copy_(wl.dev[i]["dw"], non_blocking=True)
                    wl.host[i]["db"].copy_(wl.dev[i]["db"], non_blocking=True)

        def e2e_body():
            # fork: the copy streams start after everything already on `stream`
            up.wait_stream(stream)
            down.wait_stream(stream)
            with torch.cuda.stream(up):
                for i, (h, d) in enumerate(zip(wl.host, wl.dev)):
                    for k in wl.inputs(h):
                        if k != "dy":
                            d[k].copy_(h[k], non_blocking=True)
                    ev_fwd_in[i].record(up)
                for i in reversed(range(nl)):
                    wl.dev[i]["dy"].copy_(wl.host[i]["dy"], non_blocking=True)
                    ev_dy_in[i].record(up)
            with torch.cuda.stream(stream):
                run_step(wl, sh, record=hook, interleave=True)
            # join: `stream` ends after the last download
            stream.wait_stream(down)
            stream.wait_stream(up)

        # The same step, host copies included, as one CUDA graph (memcpy nodes
        # from the pinned host buffers, the C ABI kernels, cross-stream event
        # edges) so that host-side launch overhead does not pace it.
        e2e_graph = None
        if graph is not None:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph, stream=stream):
                e2e_body()
            torch.cuda.synchronize(device)

        def e2e_step():
            with torch.cuda.stream(stream):
                if e2e_graph is not None:
                    e2e_graph.replay()
                else:
                    e2e_body()
            stream.synchronize()
        e2e_step()
        n_e2e = max(3, min(args.steps, 10))
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        # each step timed on its own (it ends with a synchronize); the median
        # step is reported, since the host link is shared with the rest of the
        # machine and single steps can stall on it
        step_ms = []
        for _ in range(n_e2e):
            t0 = time.perf_counter()
            e2e_step()
            step_ms.append((time.perf_counter() - t0) * 1e3)
        e2e_ms = max_over_ranks(float(np.median(step_ms)), ws, device)
        e2e = {"value": round(flops_step * ws / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "ms_per_step": round(e2e_ms, 3), "steps": n_e2e, "statistic": "median step",
               "ms_min_max": [round(min(step_ms), 3), round(max(step_ms), 3)],
               "launch": "stream" if e2e_graph is None else "CUDA graph (copies + C ABI calls)",
               "h2d_bytes_per_step": wl.h2d_bytes(), "d2h_bytes_per_step": wl.d2h_bytes()}

    gates = None
    if not args.no_gates:
        gates = config_gates(args.seed, device, stream, flush, peaks)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(layers, args.seed, budget_s=args.cpu_budget)

    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 + Box-Muller normals; no dataset, no trained weights)",
        "config": {"workload": args.workload, "layers": len(layers), "batch": layers[0].N,
                   "layout": "NHWC bf16 activations, KRSC bf16 weights, fp32 accumulate",
                   "l2": FLUSH_NOTE,
                   "flops_per_step": flops_step, "flops_per_step_padded_cin": flops_padded,
                   "launch": "stream" if graph is None else "CUDA graph of the step's C ABI calls",
                   "kernel_family": args.path,
                   "fused_act_backward": bool(args.fused_act),
                   "concat_free_up_path": bool(args.concat_free),
                   "wgrad_streams": 1 if wstreams is None else len(wstreams)},
        "pct_of_roofline": round(roof_s / (ms * 1e-3), 4),
        "roofline": {"bound": "tensor",
                     "kernel": {"fwd": "k_igemm + k_igemm_pair + k_stem_fwd (forward pass)",
                                "dgrad": "k_igemm + k_igemm_pair + k_stem_dgrad (dgrad pass)",
                                "wgrad": "k_wgrad + k_wgrad_c8 + k_wgrad_reduce (wgrad pass)"}[dom],
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "frac_burst": round(achieved / peaks["bf16_tflops"], 4),
                     "frac_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                     "peak_source": "%s %s (%s)" % (
                         peaks["source"], "bf16 burst" if peak_key == "bf16_tflops" else
                         "bf16 sustained", "short timed region at full SM clock"
                         if peak_key == "bf16_tflops" else "long or throttled timed region"),
                     "traffic": recorded_pass_traffic(args.workload, dom, args.fused_act,
                                                      args.concat_free, args.path),
                     "traffic_note": "DRAM bytes of the pass's launches per step from one scoped "
                                     "ncu capture of a whole step (one pass per launch, caches "
                                     "flushed before each; writes still in L2 at a launch's end "
                                     "not counted); per-call figures of the per-layer configs "
                                     "are in gates"},
        "passes": fam,
        "gpu_launches": launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "layers_detail": per_layer,
        "gates": gates,
    }
    return line


# ---------------------------------------------------------------------------
# filtered resampling (upfirdn2d) between the UNet's levels
# ---------------------------------------------------------------------------
UFD_METRIC = "upfirdn2d UNet 2x resampling throughput (GB/s of algorithmic HBM traffic) on 1 GB300 and % of HBM roofline"


def upfirdn2d_arm(args):
    """One step = the six resampling ops between the UNet's levels (2x down at
    64, 32, 16; 2x up at 8, 16, 32), batch 64, bf16 NHWC, each through the
    upfirdn2d C ABI call.  The metric is algorithmic bytes (x read once, y
    written once) per second against the measured HBM copy bandwidth."""
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    import __graft_entry__ as ge
    ge.build()
    from x3_convolution_gb300 import _lib as Lb
    ops_ = synth.UPFIRDN2D
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=device)
    sh = stream.cuda_stream
    xs, ys, fs, hx, hy = [], [], [], [], []
    for i, op in enumerate(ops_):
        x = synth.make_resample_input(op, seed=args.seed, index=i)
        t = torch.from_numpy(synth.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
        xs.append(t.to(device))
        ys.append(torch.empty((op.N, op.Ho, op.Wo, op.C), dtype=torch.bfloat16, device=device))
        fs.append(op.filter())
        if not args.no_e2e:
            hx.append(t.pin_memory())
            hy.append(torch.empty((op.N, op.Ho, op.Wo, op.C), dtype=torch.bfloat16).pin_memory())
    bytes_step = sum(op.bytes() for op in ops_)
    flush = L2Flush(device)

    def call(i, x=None, y=None):
        op = ops_[i]
        Lb.upfirdn2d(xs[i] if x is None else x, fs[i], ys[i] if y is None else y, op.N, op.C, op.H,
                     op.W, op.up, op.down, *op.pad, 4, 4, Lb.DT_BF16, sh)

    def step():
        for i in range(len(ops_)):
            call(i)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(gpu_selector(device))
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    evs = []
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    ms_max = max_over_ranks(ms, ws, device)
    value = bytes_step * ws / (ms_max * 1e-3) / 1e9
    # each op timed alone (L2 flushed before every call)
    detail = []
    for i, op in enumerate(ops_):
        us = call_us(stream, flush, lambda i=i: call(i))
        detail.append({"name": op.name, "C": op.C, "H": op.H, "Ho": op.Ho, "up": op.up, "down": op.down,
                       "us": round(us, 2), "gbs": round(op.bytes() / (us * 1e-6) / 1e9, 1),
                       "frac": round(op.bytes() / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3)})
    dom = max(detail, key=lambda d: d["us"])
    e2e = None
    if not args.no_e2e:
        def e2e_step():
            with torch.cuda.stream(stream):
                for i in range(len(ops_)):
                    xs[i].copy_(hx[i], non_blocking=True)
                    call(i)
                    hy[i].copy_(ys[i], non_blocking=True)
            stream.synchronize()
        e2e_step()
        t = []
        for _ in range(max(3, min(args.steps, 10))):
            t0 = time.perf_counter()
            e2e_step()
            t.append((time.perf_counter() - t0) * 1e3)
        e_ms = max_over_ranks(float(np.median(t)), ws, device)
        e2e = {"value": round(bytes_step * ws / (e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
               "ms_per_step": round(e_ms, 3), "statistic": "median step",
               "h2d_bytes_per_step": sum(h.numel() * 2 for h in hx),
               "d2h_bytes_per_step": sum(h.numel() * 2 for h in hy)}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = upfirdn2d_cpu_baseline(args.seed, budget_s=args.cpu_budget)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        return None
    achieved = value / ws
    return {
        "metric": UFD_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 + Box-Muller normals)",
        "config": {"workload": "upfirdn2d", "ops": len(ops_), "batch": ops_[0].N,
                   "filter": "binomial [1,3,3,1] x [1,3,3,1] / 64 (x up^2 when upsampling)",
                   "bytes_per_step": bytes_step, "l2": FLUSH_NOTE},
        "roofline": {"bound": "hbm", "kernel": "k_upfirdn2d (all six ops)",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": (RECORDED_UFD_TRAFFIC
                                 if sources_sha256(UFD_SOURCES) == UFD_SHA256 else None),
                     "traffic_note": "DRAM bytes of the six ops per step from one scoped ncu "
                                     "capture (caches flushed before each op; outputs still in "
                                     "L2 at an op's end not counted)",
                     "peak_source": peaks["source"] + " HBM copy"},
        "ops_detail": detail, "slowest_op": dom["name"],
        "gpu_launches": len(ops_) * args.steps, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
    }


def upfirdn2d_cpu_baseline(seed, budget_s=None):
    """The oracle on one image of each op (fp64, all host cores), in bytes/s.
    Without a budget: one pass over the six ops.  With one: passes over the
    ops (image 0 of each) repeat until the budget is spent."""
    import oracle
    tot_t, tot_b, passes = 0.0, 0, 0
    while True:
        for i, op in enumerate(synth.UPFIRDN2D):
            one = synth.Resample(op.name, 1, op.C, op.H, op.W, op.up, op.down, op.pad)
            x = synth.make_resample_input(one, seed=seed, index=i)
            t0 = time.perf_counter()
            oracle.upfirdn2d(x, one.filter().astype(np.float64), one.up, one.down, one.pad)
            tot_t += time.perf_counter() - t0
            tot_b += one.bytes()
        passes += 1
        if budget_s is None or tot_t >= budget_s:
            break
    return {"value": tot_b / tot_t / 1e9, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": "%d pass(es) over image 0 of each of %d ops (fp64, four materialised steps), %.2f s"
                      % (passes, len(synth.UPFIRDN2D), tot_t)}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(L: synth.Layer, seed: int, index: int):
    """fwd + dgrad + wgrad of the first image of layer L; returns (seconds, flops)."""
    import oracle
    L1 = synth.Layer(L.name, 1, L.Cin, L.Cout, L.H, L.W, act=L.act, cin_real=L.cin_real,
                     dtype=L.dtype, stride=L.stride)
    t = synth.make_tensors(L1, seed=seed, index=index)
    x, w, b, dy = (np.asarray(a, np.float64) for a in (t.x, t.w, t.bias, t.dy))
    t0 = time.perf_counter()
    if L.stride == 1:
        oracle.conv3x3_fwd(x, w, b, L.act)
        oracle.conv3x3_dgrad(dy, w)
        oracle.conv3x3_wgrad(x, dy)
    else:
        oracle.conv3x3_fwd_strided(x, w, b, L.act, u=L.stride)
        oracle.conv3x3_dgrad_strided(dy, w, L.H, L.W, u=L.stride)
        oracle.conv3x3_wgrad_strided(x, dy, u=L.stride)
    dt = time.perf_counter() - t0
    return dt, 3 * L1.flops_per_pass()


def cpu_baseline(layers, seed, budget_s=10.0):
    """The oracle's fwd + dgrad + wgrad on image 0 of each layer (fp64, all host
    cores), cheapest layers first, in passes over the layers until the budget
    (seconds of CPU work) is spent; a pass stops early once it is."""
    import oracle
    tot_t, tot_f, calls, passes = 0.0, 0, 0, 0
    order = sorted(range(len(layers)), key=lambda i: layers[i].flops_per_pass() / layers[i].N)
    while tot_t < budget_s:
        passes += 1
        for i in order:
            if tot_t >= budget_s:
                break
            dt, fl = oracle_sample(layers[i], seed, i)
            tot_t += dt
            tot_f += fl
            calls += 1
    return {"value": tot_f / tot_t / 1e12, "unit": UNIT, "cores": oracle.threads(),
            "kind": "oracle",
            "sample": "fwd+dgrad+wgrad of image 0 of a layer, %d layer samples over %d of %d layers "
                      "in %d pass(es) (fp64 loop nests), %.1f s"
                      % (calls, min(calls, len(layers)), len(layers), passes, tot_t)}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    synth.build()
    if args.workload == "upfirdn2d":
        steps = []
        for _ in range(args.warmup):
            upfirdn2d_cpu_baseline(args.seed)
        for _ in range(args.steps):
            steps.append(upfirdn2d_cpu_baseline(args.seed))
        value = float(np.mean([c["value"] for c in steps]))
        return {
            "impl": "reference", "metric": UFD_METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "upfirdn2d", "ops": len(synth.UPFIRDN2D)},
            "cpu_baseline": dict(steps[-1], value=value),
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    layers = synth.CONFIGS[args.workload]
    for i in range(args.warmup):
        oracle_sample(layers[i % len(layers)], args.seed, i % len(layers))
    tt, tf = 0.0, 0
    per = []
    for s in range(args.steps):
        i = s % len(layers)
        dt, fl = oracle_sample(layers[i], args.seed, i)
        tt += dt
        tf += fl
        per.append(dt)
    value = tf / tt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "layers": len(layers),
                                        "batch": layers[0].N},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": "each step: fwd+dgrad+wgrad of image 0 of one layer, cycling "
                                   "through the %d layers" % len(layers)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", choices=sorted(synth.CONFIGS) + ["upfirdn2d"], default="unet")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-detail", action="store_true",
                    help="omit the per-layer breakdown of the step (extra untimed steps)")
    ap.add_argument("--no-gates", action="store_true",
                    help="omit the per-config calls timed alone against their targets")
    ap.add_argument("--wgrad-streams", type=int, default=2,
                    help="streams the wgrad calls go round-robin over (1 = one stream)")
    ap.add_argument("--path", choices=["auto", "tensor", "simt"], default="auto",
                    help="kernel family of the plain calls (auto: the library picks)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps call by call instead of replaying a CUDA graph")
    ap.add_argument("--concat-free", action="store_true",
                    help="up-path convs take main and skip as two tensors (no concat buffer)")
    ap.add_argument("--fused-act", action="store_true",
                    help="training-step variant: forwards also store z, dgrads take the input's "
                         "pre-activation and return the gradient through its activation")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.wgrad_streams < 1:
        ap.error("--wgrad-streams must be >= 1")
    if args.impl == "reference":
        line = reference_arm(args)
    elif args.workload == "upfirdn2d":
        line = upfirdn2d_arm(args)
    else:
        line = cuda_arm(args)
    if line is not None:
        if line.get("layers_detail") is None:
            line.pop("layers_detail", None)
        print(json.dumps(line), flush=True)
    ws, _, _ = dist_env()
    if ws > 1 and args.impl == "cuda":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
