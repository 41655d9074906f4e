"""Shared test helpers: tolerances, numpy <-> torch transfers of half-precision
bit patterns, guard-banded output buffers."""
from __future__ import annotations

import numpy as np

# Tolerances of the parity contract:
#  - fp32 outputs: max_i |y_i - r_i| / max(|r_i|, rms(r)) <= 1e-3
#  - fp16 / bf16 outputs: |y - r| <= 1e-2 + 2e-2 max(|r|, rms(r)) elementwise
F32_TOL = 1e-3
HALF_ATOL, HALF_RTOL = 1e-2, 2e-2
TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}
CODE = {"f32": 0, "f16": 1, "bf16": 2}
SENTINEL = 0x5A


def f32_error(y, ref) -> float:
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    denom = np.maximum(np.abs(ref), rms)
    denom = np.where(denom == 0, 1.0, denom)
    return float(np.max(np.abs(y - ref) / denom)) if ref.size else 0.0


def assert_f32_close(y, ref, tol=F32_TOL):
    err = f32_error(y, ref)
    assert err <= tol, f"fp32 relative error {err:.3g} > {tol}"


def assert_half_close(y, ref):
    """|y - r| <= 1e-2 + 2e-2 * max(|r|, rms(r)) elementwise.  The relative part is
    measured against max(|r_i|, rms(r)), as in the fp32 rule: rounding a dequantised
    weight to a 16-bit tensor-core operand gives errors that scale with the output's
    rms, so an exact product of bf16-rounded weights already exceeds 2e-2 |r_i| on
    near-zero outputs at K = 2048."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bad = np.abs(y - ref) > HALF_ATOL + HALF_RTOL * np.maximum(np.abs(ref), rms)
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} half-precision outputs out of tolerance; "
                           f"worst |y-r| = {np.max(np.abs(y - ref)):.3g}")


def assert_close(y, ref, dtype: str):
    if dtype == "f32":
        assert_f32_close(y, ref)
    else:
        assert_half_close(y, ref)


def to_dev(a: np.ndarray, dtype: str | None = None):
    """numpy -> contiguous CUDA tensor.  uint16 arrays with dtype f16/bf16 are bit patterns."""
    import torch
    a = np.ascontiguousarray(a)
    if dtype in ("f16", "bf16"):
        t = torch.from_numpy(a.view(np.int16)).view(torch.float16 if dtype == "f16" else torch.bfloat16)
    elif a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def to_f64(t) -> np.ndarray:
    """CUDA/CPU tensor of any float dtype -> float64 numpy (exact widening)."""
    return t.detach().double().cpu().numpy()


def empty_guarded(n: int, dtype: str, guard: int = 64):
    """A flat CUDA buffer of n elements with `guard` sentinel bytes on both sides.
    Returns (inner view, full byte buffer)."""
    import torch
    tdt = getattr(torch, TORCH_DT[dtype])
    esz = torch.tensor([], dtype=tdt).element_size()
    full = torch.full((n * esz + 2 * guard,), SENTINEL, dtype=torch.uint8, device="cuda")
    inner = full[guard:guard + n * esz].view(tdt)
    return inner, full


def guards_intact(full, guard: int = 64) -> bool:
    h = full.cpu().numpy()
    return bool((h[:guard] == SENTINEL).all() and (h[-guard:] == SENTINEL).all())
