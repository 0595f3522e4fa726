"""Helpers for the GPU parity tests: device copies of seeded inputs and the
error metrics the tolerances are written against."""
from __future__ import annotations

import numpy as np
import torch

import synth


def to_dev_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 array holding bf16-representable values -> contiguous bf16 CUDA tensor (exact)."""
    bits = synth.bf16_bits(a)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    """max_i |got_i - ref_i| / max_i |ref_i| (the parity metric)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significand bits)."""
    a = np.abs(np.asarray(v, np.float64))
    a = np.maximum(a, 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_bf16_store(got_bf16, ref, tol=2e-3):
    """|y - ref| <= ulp_bf16(ref)/2 + tol * max|ref|, elementwise (one rounding on store)."""
    got = np.asarray(got_bf16, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = 0.5 * ulp_bf16(ref) + tol * np.max(np.abs(ref))
    bad = np.abs(got - ref) > bound
    return int(bad.sum())


def rne_bf16(a32: np.ndarray) -> np.ndarray:
    return synth.bf16_round(np.asarray(a32, np.float32)).astype(np.float64)
