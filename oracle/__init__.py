"""The oracle -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around ``oracle.c``: a plain fp64 CPU restatement of
block-quantized weight-only matmul (MatMulNBits) and of the QMoE expert FFN.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it imports nothing from the library.

Arrays are numpy.  Half-precision inputs are passed as their raw bit patterns
(``uint16`` arrays, or ``float16`` arrays which are reinterpreted); ``dtype``
arguments are one of ``"f32"``, ``"f16"``, ``"bf16"``.

Every function is pinned by ``tests/test_oracle_pins.py`` against hand-derived
byte vectors, brute-force expansion, closed forms and invariants.  SwiGLU is
the one step whose parity is unpinned beyond its definition silu(g) * u.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
FC1_LAYOUTS = {"interleaved": 0, "concat": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with the host gcc.

    -ffp-contract=off keeps every multiply and add separately rounded, so the
    fp64 sums are identical on x86-64 and AArch64.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            C = ctypes.c_int
            sig = {
                "orc_unpack_codes": [P, I64, I64, C, C, P],
                "orc_pack_codes": [P, I64, I64, C, C, P],
                "orc_unpack_zero_points": [P, I64, I64, C, P],
                "orc_pack_zero_points": [P, I64, I64, C, P],
                "orc_dequantize": [P, P, C, P, I64, I64, C, C, P],
                "orc_mnb_matmul": [P, C, I64, I64, P, P, C, P, I64, C, C, P, I64, P, C],
                "orc_route": [P, I64, I64, C, C, P, P],
                "orc_permute": [P, I64, C, I64, P, P, P],
                "orc_qmoe": [P, C, I64, I64, P, I64, C, C, P, P, P, C, P, P, P, C, I64, C, C, P,
                             I64, P, C],
                "orc_qmoe_ex": [P, C, I64, I64, P, C, I64, C, C, P, P, P, P, C, P, P, P, P, C, P, C, I64, C, C,
                                P, I64, P, C],
                "orc_quantize_int3": [P, C, I64, I64, C, C, P, P, P],
                "orc_quantize_a_int8": [P, C, I64, I64, C, P, P],
                "orc_gate_up_swiglu": [P, C, I64, I64, P, P, C, P, I64, C, C, C, P, C],
                "orc_mnb_matmul_int8a": [P, C, I64, I64, P, P, C, P, I64, C, C, P, C],
                "orc_round_to_half_bits": [P, I64, C, P],
                "orc_prepack": [P, P, C, P, I64, I64, C, C, ctypes.c_uint64, P],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = C
            lib.orc_prepack_size.argtypes = [I64, I64, C, C, C, C]
            lib.orc_prepack_size.restype = I64
            _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _elem(a, dtype: str):
    """Contiguous array with the element width `dtype` names (no value change)."""
    if dtype == "f32":
        return _c(a, np.float32)
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize != 2:
        raise TypeError(f"{dtype} data must be passed as 16-bit patterns, got {a.dtype}")
    return a.view(np.uint16)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments")


def n_blocks(K: int, bs: int) -> int:
    return (K + bs - 1) // bs


def row_bytes(K: int, bits: int, bs: int) -> int:
    return n_blocks(K, bs) * bs * bits // 8


def zp_row_bytes(nb: int, bits: int) -> int:
    return (nb * bits + 7) // 8


def unpack_codes(packed, rows: int, K: int, bits: int, bs: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    assert packed.size >= rows * row_bytes(K, bits, bs)
    out = np.zeros((rows, K), np.uint8)
    _check(_lib().orc_unpack_codes(_ptr(packed), rows, K, bits, bs, _ptr(out)), "unpack")
    return out


def pack_codes(codes, bits: int, bs: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    rows, K = codes.shape
    out = np.zeros((rows, row_bytes(K, bits, bs)), np.uint8)
    _check(_lib().orc_pack_codes(_ptr(codes), rows, K, bits, bs, _ptr(out)), "pack")
    return out


def unpack_zero_points(zp, rows: int, nb: int, bits: int) -> np.ndarray:
    zp = _c(zp, np.uint8)
    out = np.zeros((rows, nb), np.uint8)
    _check(_lib().orc_unpack_zero_points(_ptr(zp), rows, nb, bits, _ptr(out)), "unpack zp")
    return out


def pack_zero_points(zcodes, bits: int) -> np.ndarray:
    zcodes = _c(zcodes, np.uint8)
    rows, nb = zcodes.shape
    out = np.zeros((rows, zp_row_bytes(nb, bits)), np.uint8)
    _check(_lib().orc_pack_zero_points(_ptr(zcodes), rows, nb, bits, _ptr(out)), "pack zp")
    return out


def dequantize(packed, scales, s_dtype: str, zp, N: int, K: int, bits: int, bs: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    scales = _elem(scales, s_dtype)
    zp = _c(zp, np.uint8)
    out = np.zeros((N, K), np.float64)
    _check(_lib().orc_dequantize(_ptr(packed), _ptr(scales), DTYPES[s_dtype], _ptr(zp), N, K, bits,
                                 bs, _ptr(out)), "dequantize")
    return out


def mnb_matmul(A, a_dtype: str, packed, scales, s_dtype: str, zp, N: int, K: int, bits: int,
               bs: int, mrows=None, threads: int = 1) -> np.ndarray:
    """fp64 Y[len(mrows) or M, N]; A is [M, K] in a_dtype."""
    A = _elem(A, a_dtype)
    M = A.size // K if K else 0
    packed = _c(packed, np.uint8)
    scales = _elem(scales, s_dtype)
    zp = _c(zp, np.uint8)
    rows = None if mrows is None else np.ascontiguousarray(mrows, dtype=np.int64)
    n_rows = M if rows is None else rows.size
    out = np.zeros((n_rows, N), np.float64)
    _check(_lib().orc_mnb_matmul(_ptr(A), DTYPES[a_dtype], M, K, _ptr(packed), _ptr(scales),
                                 DTYPES[s_dtype], _ptr(zp), N, bits, bs, _ptr(rows),
                                 0 if rows is None else rows.size, _ptr(out), threads), "matmul")
    return out


def quantize_a_int8(A, a_dtype: str, K: int, bs: int):
    """Per-(row, block) symmetric int8 quantisation of activations A [M, K]:
    (aq int8 [M, K], sa float32 [M, nb]) -- the accuracy_level=4 activation step."""
    A = _elem(A, a_dtype)
    M = A.size // K
    nb = n_blocks(K, bs)
    aq = np.zeros((M, K), np.int8)
    sa = np.zeros((M, nb), np.float32)
    _lib().orc_quantize_a_int8(_ptr(A), DTYPES[a_dtype], M, K, bs, _ptr(aq), _ptr(sa))
    return aq, sa


def mnb_matmul_int8a(A, a_dtype: str, packed, scales, s_dtype: str, zp, N: int, K: int, bits: int, bs: int,
                     threads: int = 1) -> np.ndarray:
    """fp64 Y[M, N] of MatMulNBits with int8 activation compute (accuracy_level=4)."""
    A = _elem(A, a_dtype)
    M = A.size // K if K else 0
    packed = _c(packed, np.uint8)
    scales = _elem(scales, s_dtype)
    zp = _c(zp, np.uint8)
    out = np.zeros((M, N), np.float64)
    _check(_lib().orc_mnb_matmul_int8a(_ptr(A), DTYPES[a_dtype], M, K, _ptr(packed), _ptr(scales),
                                       DTYPES[s_dtype], _ptr(zp), N, bits, bs, _ptr(out), threads), "matmul_int8a")
    return out


def gate_up_swiglu(A, a_dtype: str, packed, scales, s_dtype: str, zp, I: int, K: int, bits: int, bs: int,
                   layout: str = "interleaved", threads: int = 1) -> np.ndarray:
    """fp64 H[M, I] = silu(A . Wg^T) * (A . Wu^T), gate/up rows of packed [2I, ...] in `layout`."""
    A = _elem(A, a_dtype)
    M = A.size // K if K else 0
    packed = _c(packed, np.uint8)
    scales = _elem(scales, s_dtype)
    zp = _c(zp, np.uint8)
    out = np.zeros((M, I), np.float64)
    _check(_lib().orc_gate_up_swiglu(_ptr(A), DTYPES[a_dtype], M, K, _ptr(packed), _ptr(scales), DTYPES[s_dtype],
                                     _ptr(zp), I, bits, bs, FC1_LAYOUTS[layout], _ptr(out), threads), "gate_up_swiglu")
    return out


def prepack(packed, scales, s_dtype: str, zp, N: int, K: int, bits: int, bs: int, identity: int = 0) -> np.ndarray:
    """The library's version-1 prepacked bytes (header + rows) of a row-local weight."""
    packed = _c(packed, np.uint8)
    scales = _elem(scales, s_dtype)
    zp = _c(zp, np.uint8)
    n = _lib().orc_prepack_size(N, K, bits, bs, DTYPES[s_dtype], int(zp is not None))
    out = np.zeros(n, np.uint8)
    _check(_lib().orc_prepack(_ptr(packed), _ptr(scales), DTYPES[s_dtype], _ptr(zp), N, K, bits, bs,
                              ctypes.c_uint64(identity), _ptr(out)), "prepack")
    return out


def route(logits, k: int, normalize: bool = True):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    _check(_lib().orc_route(_ptr(logits), T, E, k, int(bool(normalize)), _ptr(idx), _ptr(w)), "route")
    return idx, w


def permute(idx, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    _check(_lib().orc_permute(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm)), "permute")
    return counts, offsets, perm


def qmoe(X, act_dtype: str, logits, k: int, normalize: bool, fc1_w, fc1_scales, fc1_zp,
         fc1_bits: int, fc2_w, fc2_scales, fc2_zp, fc2_bits: int, I: int, bs: int,
         fc1_layout: str = "interleaved", tokens=None, threads: int = 1) -> np.ndarray:
    """fp64 Y[len(tokens) or T, H]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    X = _elem(X, act_dtype)
    H = X.size // T
    toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    rows = T if toks is None else toks.size
    out = np.zeros((rows, H), np.float64)
    # converted inputs stay referenced until the call returns
    keep = [_c(fc1_w, np.uint8), _elem(fc1_scales, act_dtype), _c(fc1_zp, np.uint8),
            _c(fc2_w, np.uint8), _elem(fc2_scales, act_dtype), _c(fc2_zp, np.uint8)]
    args = (_ptr(X), DTYPES[act_dtype], T, H, _ptr(logits), E, k, int(bool(normalize)),
            _ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]), fc1_bits, _ptr(keep[3]), _ptr(keep[4]),
            _ptr(keep[5]), fc2_bits, I, bs, FC1_LAYOUTS[fc1_layout], _ptr(toks),
            0 if toks is None else toks.size, _ptr(out), threads)
    _check(_lib().orc_qmoe(*args), "qmoe")
    return out


def qmoe_ex(X, act_dtype: str, logits, logits_dtype: str, k: int, normalize: bool, fc1_w, fc1_scales, fc1_zp,
            fc1_bias, fc1_bits: int, fc2_w, fc2_scales, fc2_zp, fc2_bias, fc2_bits: int, I: int, bs: int,
            fc1_layout: str = "interleaved", agg=None, agg_dtype: str = "f32", tokens=None,
            threads: int = 1) -> np.ndarray:
    """fp64 Y[len(tokens) or T, H] with the optional inputs: logits [T, E] in
    logits_dtype, fc1_bias [E, 2I] and fc2_bias [E, H] in act_dtype (or None),
    agg [T, E] aggregation weights in agg_dtype (or None)."""
    L = _elem(logits, logits_dtype)
    T, E = np.asarray(logits).shape
    X = _elem(X, act_dtype)
    H = X.size // T
    toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    rows = T if toks is None else toks.size
    out = np.zeros((rows, H), np.float64)
    keep = [_c(fc1_w, np.uint8), _elem(fc1_scales, act_dtype), _c(fc1_zp, np.uint8),
            None if fc1_bias is None else _elem(fc1_bias, act_dtype),
            _c(fc2_w, np.uint8), _elem(fc2_scales, act_dtype), _c(fc2_zp, np.uint8),
            None if fc2_bias is None else _elem(fc2_bias, act_dtype),
            None if agg is None else _elem(agg, agg_dtype)]
    args = (_ptr(X), DTYPES[act_dtype], T, H, _ptr(L), DTYPES[logits_dtype], E, k, int(bool(normalize)),
            _ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]), _ptr(keep[3]), fc1_bits, _ptr(keep[4]), _ptr(keep[5]),
            _ptr(keep[6]), _ptr(keep[7]), fc2_bits, _ptr(keep[8]), DTYPES[agg_dtype], I, bs,
            FC1_LAYOUTS[fc1_layout], _ptr(toks), 0 if toks is None else toks.size, _ptr(out), threads)
    _check(_lib().orc_qmoe_ex(*args), "qmoe_ex")
    return out


def quantize_int3(W, w_dtype: str, bs: int, s_dtype: str):
    """Symmetric grouped INT3 round-to-nearest of W [N, K] (K % bs == 0).

    Returns (packed uint8 [N, K/bs * 3*bs/8], scales [N, K/bs], bad bool [N, K/bs]):
    scales are float32 for "f32" and raw uint16 bit patterns for "f16" / "bf16";
    bad marks the rejected blocks (non-finite weight or stored scale, or a
    nonzero block whose stored scale rounds to zero)."""
    W = _elem(W, w_dtype)
    N, K = W.shape
    nb = K // bs
    packed = np.zeros((N, nb * bs * 3 // 8), np.uint8)
    scales = np.zeros((N, nb), np.float32 if s_dtype == "f32" else np.uint16)
    bad = np.zeros((N, nb), np.uint8)
    _check(_lib().orc_quantize_int3(_ptr(W), DTYPES[w_dtype], N, K, bs, DTYPES[s_dtype], _ptr(packed),
                                    _ptr(scales), _ptr(bad)), "quantize_int3")
    return packed, scales, bad.astype(bool)


def round_to_half_bits(x, dtype: str) -> np.ndarray:
    """binary32 values -> the bit patterns the quantizer stores for dtype
    "f16" or "bf16" (round to nearest, ties to even)."""
    x = _c(np.asarray(x, np.float32).reshape(-1), np.float32)
    out = np.zeros(x.size, np.uint16)
    _check(_lib().orc_round_to_half_bits(_ptr(x), x.size, 1 if dtype == "bf16" else 0, _ptr(out)), "round")
    return out
