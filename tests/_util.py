"""Shared test helpers: tolerances, numpy <-> torch transfers of half-precision
bit patterns, guard-banded output buffers."""
from __future__ import annotations

import numpy as np

# Tolerances of the parity contract:
#  - fp32 outputs: max_i |y_i - r_i| / max(|r_i|, rms(r)) <= 1e-3
#  - fp16 / bf16 outputs: |y_i - r_i| <= 1e-2 + 2e-2 |r_i| elementwise
#  - bf16 outputs of the tensor-core paths only (bf16 activations, so the
#    dequantised weight is a bf16 MMA operand): |y_i - r_i| <= 1e-2 + 2e-2
#    max(|r_i|, rms(r)), and the number of outputs outside the elementwise
#    rule is printed.  An exact product of bf16-rounded weights already
#    misses the elementwise rule on a fraction of a percent of the near-zero
#    outputs at K = 2048.
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


def half_violations(y, ref) -> int:
    """Outputs outside the elementwise 16-bit rule |y - r| <= 1e-2 + 2e-2 |r|."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return int(np.sum(np.abs(y - ref) > HALF_ATOL + HALF_RTOL * np.abs(ref)))


def assert_half_close(y, ref):
    """|y - r| <= 1e-2 + 2e-2 |r|, every output."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    bad = half_violations(y, ref)
    assert bad == 0, (f"{bad} of {y.size} half-precision outputs out of tolerance; "
                      f"worst |y-r| = {np.max(np.abs(y - ref)):.3g}")


def assert_bf16_tc_close(y, ref, label: str = ""):
    """bf16 tensor-core outputs: |y - r| <= 1e-2 + 2e-2 max(|r|, rms(r)) every
    output; prints how many outputs miss the elementwise rule."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    elementwise = half_violations(y, ref)
    print(f"[bf16 tensor-core rule] {label}: {elementwise} of {y.size} outputs outside the elementwise rule "
          f"({100.0 * elementwise / max(y.size, 1):.3f} %)")
    bad = np.abs(y - ref) > HALF_ATOL + HALF_RTOL * np.maximum(np.abs(ref), rms)
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} bf16 outputs out of tolerance; "
                           f"worst |y-r| = {np.max(np.abs(y - ref)):.3g}")


def _swiglu_parts(g, u):
    """h = silu(g) u, silu'(g), and the rms of g and u."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    sig = 1.0 / (1.0 + np.exp(-g))
    h = g * sig * u
    dsilu = sig * (1.0 + g * (1.0 - sig))
    return g, u, h, dsilu, float(np.sqrt(np.mean(g * g))), float(np.sqrt(np.mean(u * u)))


def swiglu_f32_error(y, g, u) -> float:
    """The fp32 rule carried through h = silu(g) * u: the gate and up products may
    each miss by F32_TOL of max(|value|, its rms), so h may miss by
    |silu'(g)| |u| dg + |silu(g)| du to first order.  Returns max |y - h| over
    that allowance (at 1x the rule); the floor keeps outputs where every term
    vanishes from dividing by zero."""
    y = np.asarray(y, np.float64)
    if y.size == 0:
        return 0.0
    g, u, h, dsilu, rg, ru = _swiglu_parts(g, u)
    allow = np.abs(dsilu * u) * np.maximum(np.abs(g), rg) + np.abs(g / (1.0 + np.exp(-g))) * np.maximum(np.abs(u), ru)
    allow = allow + 1e-2 * rg * ru
    return float(np.max(np.abs(y - h) / allow))


def assert_swiglu_bf16_tc_close(y, g, u, label: str = ""):
    """bf16 tensor-core SwiGLU outputs: the bf16 tensor-core rule on the gate and up
    products (|d| <= 1e-2 + 2e-2 max(|value|, rms)) carried through silu(g) * u to
    first order, plus the rounding of h to bf16 (2^-8 |h|).  Prints how many
    outputs miss the plain elementwise 16-bit rule on h."""
    y = np.asarray(y, np.float64)
    g, u, h, dsilu, rg, ru = _swiglu_parts(g, u)
    eg = HALF_ATOL + HALF_RTOL * np.maximum(np.abs(g), rg)
    eu = HALF_ATOL + HALF_RTOL * np.maximum(np.abs(u), ru)
    allow = np.abs(dsilu * u) * eg + np.abs(g / (1.0 + np.exp(-g))) * eu + 2.0 ** -8 * np.abs(h)
    elementwise = half_violations(y, h)
    print(f"[bf16 tensor-core SwiGLU rule] {label}: {elementwise} of {y.size} outputs outside the elementwise "
          f"rule ({100.0 * elementwise / max(y.size, 1):.3f} %), worst fraction of the allowance "
          f"{float(np.max(np.abs(y - h) / allow)) if y.size else 0.0:.3g}")
    bad = np.abs(y - h) > allow
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} bf16 SwiGLU outputs out of tolerance"


def assert_swiglu_f32_close(y, g, u, tol=F32_TOL, label: str = ""):
    err = swiglu_f32_error(y, g, u) * tol
    if label:
        print(f"[{label}] SwiGLU-propagated fp32 error {err:.3g} (rule {tol})")
    assert err <= tol, f"fp32 error through SwiGLU {err:.3g} > {tol}"


def assert_close(y, ref, y_dtype: str, a_dtype: str | None = None, tensor_cores: bool = False, label: str = ""):
    """The rule of the output dtype: fp32 for fp32 outputs, the elementwise 16-bit
    rule for fp16 / bf16 outputs, and the bf16 tensor-core rule for bf16 outputs
    of a tensor-core path fed bf16 activations."""
    if y_dtype == "f32":
        assert_f32_close(y, ref)
    elif tensor_cores and a_dtype == "bf16" and y_dtype == "bf16":
        assert_bf16_tc_close(y, ref, label)
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


def guarded_workspace(nbytes: int, guard: int = 256):
    """A device workspace of nbytes (256-byte aligned inside) with `guard` sentinel
    bytes on both sides.  Returns (inner view, full byte buffer); check the sentinels
    with guards_intact(full, guard)."""
    import torch
    full = torch.full((nbytes + 2 * guard,), SENTINEL, dtype=torch.uint8, device="cuda")
    return full[guard:guard + nbytes], full


def guards_intact(full, guard: int = 64) -> bool:
    h = full.cpu().numpy()
    return bool((h[:guard] == SENTINEL).all() and (h[-guard:] == SENTINEL).all())
