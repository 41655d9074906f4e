"""Pins for the oracle: it is checked against things other than itself.

- hand-derived byte/nibble vectors (tests/golden/packing_vectors.json);
- brute force: codes drawn directly, the dense matrix expanded with numpy and
  multiplied with numpy's matmul;
- exact special cases (integer data, implicit == explicit zero point, partial
  block == zero-padded K, doubling the scales doubles Y);
- every binary16 / bfloat16 pattern widened against numpy / torch;
- routing against numpy's lexsort / scipy's softmax and crafted ties;
- the expert-sorted permutation against numpy's stable argsort;
- a hand-built QMoE layer whose output has a closed form.
"""
import json
import math
import os
import struct
import zlib

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "packing_vectors.json")))


def as_f64(x, dtype):
    """Reference widening by library routines (numpy float16, torch bfloat16)."""
    if dtype == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(x, np.uint16).view(np.float16).astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(x, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


# ------------------------------------------------------------- byte vectors

@pytest.mark.parametrize("v", GOLD["int4"])
def test_int4_nibble_vectors(v):
    b = bytes.fromhex(v["bytes"])
    packed = np.zeros((1, 16), np.uint8)
    packed[0, :len(b)] = list(b)
    K = 2 * len(b)
    assert oracle.unpack_codes(packed, 1, K, 4, 32)[0].tolist() == v["codes"]
    repacked = oracle.pack_codes(np.array([v["codes"]], np.uint8), 4, 32)
    assert repacked[0, :len(b)].tobytes() == b and not repacked[0, len(b):].any()


@pytest.mark.parametrize("v", GOLD["int3"])
def test_int3_cross_byte_vectors(v):
    b = bytes.fromhex(v["bytes"])
    packed = np.zeros((1, 12), np.uint8)
    packed[0, :3] = list(b)
    assert oracle.unpack_codes(packed, 1, 8, 3, 32)[0].tolist() == v["codes"]
    repacked = oracle.pack_codes(np.array([v["codes"]], np.uint8), 3, 32)
    assert repacked[0, :3].tobytes() == b and not repacked[0, 3:].any()


@pytest.mark.parametrize("v", GOLD["zero_points"])
def test_zero_point_vectors(v):
    codes = np.array([v["codes"]], np.uint8)
    z = oracle.pack_zero_points(codes, v["bits"])
    assert z[0].tobytes() == bytes.fromhex(v["bytes"])
    assert oracle.unpack_zero_points(z, 1, len(v["codes"]), v["bits"])[0].tolist() == v["codes"]


def test_int3_rows_restart_on_a_byte():
    # K=32, bs=32: each row is one 12-byte blob; row 1 starts at byte 12.
    codes = np.zeros((2, 32), np.uint8)
    codes[1, 0] = 7
    codes[0, 31] = 5  # last code of row 0 sits in bits 93..95 of the row stream
    p = oracle.pack_codes(codes, 3, 32)
    assert p.shape == (2, 12)
    assert p[1, 0] == 0x07 and not p[1, 1:].any()
    assert p[0, 11] == 5 << 5 and not p[0, :11].any()


def test_int4_row_and_block_strides():
    # Tiny-case shape: N=128, K=256, bs=32 -> 8 blobs of 16 bytes, row stride 128 bytes.
    N, K, bs = 128, 256, 32
    packed = np.zeros((N, 128), np.uint8)
    for n in range(N):
        for b in range(8):
            packed[n, 16 * b:16 * (b + 1)] = (37 * n + 11 * b + 3) & 0xFF
    codes = oracle.unpack_codes(packed, N, K, 4, bs)
    for n in (0, 1, 77, 127):
        for k in range(K):
            v = (37 * n + 11 * (k // 32) + 3) & 0xFF
            assert codes[n, k] == (v & 0xF if k % 2 == 0 else v >> 4)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
def test_pack_unpack_roundtrip(bits, bs):
    g = wl.rng(1)
    K = 2 * bs + 13
    codes = g.integers(0, 1 << bits, size=(7, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    assert packed.shape == (7, oracle.row_bytes(K, bits, bs))
    assert np.array_equal(oracle.unpack_codes(packed, 7, K, bits, bs), codes)
    # canonical bytes survive unpack -> pack
    assert np.array_equal(oracle.pack_codes(oracle.unpack_codes(packed, 7, K, bits, bs), bits, bs), packed)


# ------------------------------------------------------ widening of scalars

def test_every_f16_pattern_widens_like_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    N = pats.size
    codes = np.full((N, 32), 9, np.uint8)  # 9 - implicit zero point 8 = 1, so w = scale
    packed = oracle.pack_codes(codes, 4, 32)
    w = oracle.dequantize(packed, pats.reshape(N, 1), "f16", None, N, 32, 4, 32)[:, 0]
    ref = pats.view(np.float16).astype(np.float64)
    assert np.array_equal(w, ref, equal_nan=True)


def test_every_bf16_pattern_widens_like_torch():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    N = pats.size
    codes = np.full((N, 32), 5, np.uint8)  # INT3: 5 - implicit 4 = 1
    packed = oracle.pack_codes(codes, 3, 32)
    w = oracle.dequantize(packed, pats.reshape(N, 1), "bf16", None, N, 32, 3, 32)[:, 0]
    assert np.array_equal(w, as_f64(pats, "bf16"), equal_nan=True)


# ------------------------------------------------------------ brute force

def _case(g, N, K, bits, bs, with_zp, s_dtype):
    nb = oracle.n_blocks(K, bs)
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    scales = wl.uniform(g, (N, nb), 0.005, 0.02, s_dtype)
    zc = g.integers(0, 1 << bits, size=(N, nb), dtype=np.uint8) if with_zp else None
    zp = oracle.pack_zero_points(zc, bits) if with_zp else None
    z = zc.astype(np.float64) if with_zp else np.full((N, nb), float(1 << (bits - 1)))
    s = as_f64(scales, s_dtype)
    W = np.repeat(s, bs, axis=1)[:, :K] * (codes.astype(np.float64) - np.repeat(z, bs, axis=1)[:, :K])
    return packed, scales, zp, W


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("a_dtype,s_dtype", [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32")])
def test_brute_force_expand_then_multiply(bits, bs, with_zp, a_dtype, s_dtype):
    g = wl.rng(zlib.crc32(repr((bits, bs, with_zp, a_dtype, s_dtype)).encode()))
    N, M = 6, 3
    K = bs + 17  # one full block plus a partial one
    packed, scales, zp, W = _case(g, N, K, bits, bs, with_zp, s_dtype)
    assert np.array_equal(oracle.dequantize(packed, scales, s_dtype, zp, N, K, bits, bs), W)
    A = wl.normal(g, (M, K), a_dtype)
    Y = oracle.mnb_matmul(A, a_dtype, packed, scales, s_dtype, zp, N, K, bits, bs)
    # the expanded product summed in ascending k (a running sum: np.cumsum adds
    # strictly left to right), so the same fp64 operations in the same order
    prod = as_f64(A, a_dtype).reshape(M, 1, K) * W.reshape(1, N, K)
    ref = np.cumsum(prod, axis=2)[:, :, -1]
    assert np.array_equal(Y, ref)


def test_selected_rows_match_full_output():
    g = wl.rng(5)
    N, K, M = 9, 96, 11
    packed, scales, _ = wl.quantized_weight(g, N, K, 4, 32)
    A = wl.normal(g, (M, K))
    full = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, N, K, 4, 32, threads=3)
    part = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, N, K, 4, 32, mrows=[10, 0, 4])
    assert np.array_equal(part, full[[10, 0, 4]])


@pytest.mark.parametrize("bits", [3, 4])
def test_integer_data_is_exact(bits):
    g = wl.rng(7)
    N, K, M, bs = 13, 2048, 2, 64
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    nb = K // bs
    zp = oracle.pack_zero_points(np.zeros((N, nb), np.uint8), bits)
    scales = np.ones((N, nb), np.float32)
    A = g.integers(-4, 5, size=(M, K)).astype(np.float32)
    Y = oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    exact = A.astype(np.int64) @ codes.astype(np.int64).T
    assert np.array_equal(Y, exact.astype(np.float64))


@pytest.mark.parametrize("bits", [3, 4])
def test_implicit_equals_explicit_midpoint(bits):
    g = wl.rng(8)
    N, K, bs = 10, 320, 32
    packed, scales, _ = wl.quantized_weight(g, N, K, bits, bs)
    nb = K // bs
    zp = oracle.pack_zero_points(np.full((N, nb), 1 << (bits - 1), np.uint8), bits)
    A = wl.normal(g, (2, K))
    a = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, N, K, bits, bs)
    b = oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    assert np.array_equal(a, b)


def test_doubling_scales_doubles_output():
    g = wl.rng(9)
    N, K = 12, 200
    packed, scales, zp = wl.quantized_weight(g, N, K, 3, 64, with_zp=True)
    A = wl.normal(g, (3, K))
    a = oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, 3, 64)
    b = oracle.mnb_matmul(A, "f32", packed, scales * np.float32(2), "f32", zp, N, K, 3, 64)
    assert np.array_equal(b, 2 * a)


@pytest.mark.parametrize("K,Kpad,bs", [(2072, 2080, 32), (2080, 2112, 64), (2080, 2176, 128)])
def test_partial_block_equals_zero_padded_k(K, Kpad, bs):
    g = wl.rng(10)
    N = 8
    packed, scales, _ = wl.quantized_weight(g, N, K, 4, bs)
    assert oracle.n_blocks(K, bs) == oracle.n_blocks(Kpad, bs)
    A = wl.normal(g, (2, K))
    Ap = np.zeros((2, Kpad), np.float32)
    Ap[:, :K] = A
    a = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, N, K, 4, bs)
    b = oracle.mnb_matmul(Ap, "f32", packed, scales, "f32", None, N, Kpad, 4, bs)
    # the padded columns hold random (non-canonical) codes; they meet zero activations
    assert np.array_equal(a, b)


# ----------------------------------------------- dense FFN gate/up with SwiGLU

@pytest.mark.parametrize("layout", ["interleaved", "concat"])
def test_gate_up_swiglu_is_swiglu_of_the_two_matmuls(layout):
    """The fused projection equals silu(gate) * up of the plain matmul's gate and up
    columns (the same fp64 sums; the exponential of libm against numpy's)."""
    g = wl.rng(41)
    M, K, I, bs, bits = 3, 160, 24, 32, 3
    packed, scales, zp = wl.quantized_weight(g, 2 * I, K, bits, bs, "bf16", with_zp=True)
    A = wl.normal(g, (M, K), "bf16")
    Hh = oracle.gate_up_swiglu(A, "bf16", packed, scales, "bf16", zp, I, K, bits, bs, layout)
    GU = oracle.mnb_matmul(A, "bf16", packed, scales, "bf16", zp, 2 * I, K, bits, bs)
    gate = GU[:, 0::2] if layout == "interleaved" else GU[:, :I]
    up = GU[:, 1::2] if layout == "interleaved" else GU[:, I:]
    assert np.allclose(Hh, gate / (1 + np.exp(-gate)) * up, rtol=1e-14, atol=1e-14)


def test_gate_up_swiglu_unit_rows_closed_form():
    """Gate row p = unit vector e_p, up row p = 2 e_p (interleaved, unit scales): the
    output is silu(a_p) * 2 a_p."""
    K = I = 32
    bits, bs = 4, 32
    z = 1 << (bits - 1)
    codes = np.full((2 * I, K), z, np.uint8)
    for p in range(I):
        codes[2 * p, p] = z + 1
        codes[2 * p + 1, p] = z + 2
    packed = oracle.pack_codes(codes, bits, bs)
    a = np.linspace(-2, 2, K).astype(np.float32).reshape(1, K)
    Hh = oracle.gate_up_swiglu(a, "f32", packed, np.ones((2 * I, 1), np.float32), "f32", None, I, K, bits, bs)
    x = a.astype(np.float64)[0]
    assert np.allclose(Hh[0], x / (1 + np.exp(-x)) * 2 * x, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("bits", [1, 2, 5, 6, 7, 8])
def test_brute_force_other_widths(bits):
    """The matmul at the widths the row-local LSB-first format allows beyond 3 and 4."""
    g = wl.rng(42 + bits)
    N, M, bs = 5, 2, 32
    K = bs + 11
    packed, scales, zp, W = _case(g, N, K, bits, bs, True, "f32")
    assert np.array_equal(oracle.dequantize(packed, scales, "f32", zp, N, K, bits, bs), W)
    A = wl.normal(g, (M, K))
    Y = oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    prod = A.astype(np.float64).reshape(M, 1, K) * W.reshape(1, N, K)
    assert np.array_equal(Y, np.cumsum(prod, axis=2)[:, :, -1])


# ------------------------------------------- int8 activation compute (accuracy_level=4)

@pytest.mark.parametrize("a_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [32, 64, 128])
def test_int8_activation_quantisation_matches_binary32_numpy(a_dtype, bs):
    """aq = rint(a / (amax / 127)) in binary32 per (row, block), clamped to +-127; a
    zero block gives scale 0 and codes 0; a partial last block uses its K entries."""
    g = wl.rng(zlib.crc32(repr(("q8", a_dtype, bs)).encode()))
    M, K = 5, 3 * bs + 17
    A = wl.normal(g, (M, K), a_dtype)
    Af = as_f64(A, a_dtype).reshape(M, K).astype(np.float32)
    Af[2, :bs] = 0.0
    A = wl.cast(Af, a_dtype)
    Af = as_f64(A, a_dtype).reshape(M, K).astype(np.float32)
    aq, sa = oracle.quantize_a_int8(A, a_dtype, K, bs)
    nb = oracle.n_blocks(K, bs)
    for b in range(nb):
        blk = Af[:, b * bs:(b + 1) * bs]
        amax = np.max(np.abs(blk), axis=1).astype(np.float32)
        s = (amax / np.float32(127.0)).astype(np.float32)
        assert np.array_equal(sa[:, b], s)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(s[:, None] != 0, np.rint(blk / s[:, None]), 0).astype(np.float32)
        assert np.array_equal(aq[:, b * bs:(b + 1) * bs], np.clip(q, -127, 127).astype(np.int8))
    assert np.all(sa[2, 0] == 0) and np.all(aq[2, :bs] == 0)


@pytest.mark.parametrize("bits", [3, 4])
def test_int8_activation_matmul_is_exact_for_127_scaled_integers(bits):
    """Activations that are integers with a block maximum of exactly 127 quantise to
    themselves (scale 1), so the int8 mode equals the exact matmul."""
    g = wl.rng(31 + bits)
    M, N, K, bs = 3, 20, 256, 64
    A = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    A[:, ::bs] = 127.0
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, with_zp=True)
    exact = oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    q8 = oracle.mnb_matmul_int8a(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    assert np.allclose(q8, exact, rtol=1e-13, atol=1e-12)


def test_int8_activation_matmul_against_quantise_then_expand():
    """Brute force: quantise A (the pinned step above), expand both operands to fp64 and
    multiply; equal to the blockwise-integer formula up to fp64 rounding."""
    g = wl.rng(33)
    M, N, K, bs, bits = 4, 9, 200, 32, 3
    A = wl.normal(g, (M, K), "bf16")
    packed, scales, _ = wl.quantized_weight(g, N, K, bits, bs, "bf16")
    aq, sa = oracle.quantize_a_int8(A, "bf16", K, bs)
    Adq = aq.astype(np.float64) * np.repeat(sa.astype(np.float64), bs, axis=1)[:, :K]
    W = oracle.dequantize(packed, scales, "bf16", None, N, K, bits, bs)
    q8 = oracle.mnb_matmul_int8a(A, "bf16", packed, scales, "bf16", None, N, K, bits, bs)
    assert np.allclose(q8, Adq @ W.T, rtol=1e-12, atol=1e-12)
    # and it stays within int8 quantisation distance of the exact result
    exact = oracle.mnb_matmul(A, "bf16", packed, scales, "bf16", None, N, K, bits, bs)
    assert np.max(np.abs(q8 - exact)) < 0.05 * np.sqrt(np.mean(exact ** 2))


# ---------------------------------------------------------------- routing

def test_route_equal_logits():
    idx, w = oracle.route(np.zeros((3, 16), np.float32), 4, True)
    assert (idx == np.arange(4)).all() and (w == 0.25).all()
    idx, w = oracle.route(np.zeros((2, 16), np.float32), 4, False)
    assert (idx == np.arange(4)).all() and (w == 1 / 16).all()


def test_route_ties_go_to_lower_index():
    logits = np.array([[1, 3, 3, 2, 3], [0, 0, -1, 0, 5]], np.float32)
    idx, _ = oracle.route(logits, 3, True)
    assert idx.tolist() == [[1, 2, 4], [4, 0, 1]]
    # -0.0 and +0.0 compare equal
    idx, _ = oracle.route(np.array([[-0.0, 0.0, -1.0]], np.float32), 2, True)
    assert idx.tolist() == [[0, 1]]


def test_route_k_equals_e_is_a_stable_descending_sort():
    g = wl.rng(11)
    logits = np.round(g.standard_normal((20, 32)) * 2).astype(np.float32)  # many ties
    idx, _ = oracle.route(logits, 32, True)
    for t in range(20):
        assert idx[t].tolist() == np.lexsort((np.arange(32), -logits[t])).tolist()


@pytest.mark.parametrize("normalize", [True, False])
def test_route_weights_against_scipy_softmax(normalize):
    g = wl.rng(12)
    logits = wl.router_logits(g, 50, 128, skew=True)
    idx, w = oracle.route(logits, 8, normalize)
    for t in range(50):
        assert len(set(idx[t].tolist())) == 8
        top = np.sort(logits[t])[::-1][:8]
        assert np.array_equal(logits[t][idx[t]], top)
        if normalize:
            ref = scipy.special.softmax(logits[t][idx[t]].astype(np.float64))
            assert abs(w[t].sum() - 1) < 1e-14
        else:
            ref = scipy.special.softmax(logits[t].astype(np.float64))[idx[t]]
        assert np.allclose(w[t], ref, rtol=1e-13, atol=0)


def test_permute_is_a_stable_expert_sort():
    g = wl.rng(13)
    T, k, E = 37, 8, 128
    idx, _ = oracle.route(wl.router_logits(g, T, E, skew=True), k, True)
    counts, offsets, perm = oracle.permute(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm, np.argsort(idx.ravel(), kind="stable"))


# ------------------------------------------------------------------- QMoE

def _unit_rows(rows, K, bits, bs, col_of_row, value=1):
    """Packed rows with code z+value at column col_of_row[r] and z elsewhere (z implicit)."""
    z = 1 << (bits - 1)
    codes = np.full((rows, K), z, np.uint8)
    for r, c in enumerate(col_of_row):
        if c is not None:
            codes[r, c] = z + value
    return oracle.pack_codes(codes, bits, bs)


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("bits", [(3, 3), (4, 3), (3, 4), (4, 4)])
def test_qmoe_hand_built_layer_closed_form(layout, bits):
    """Expert 1's FC1 gate rows are unit vectors, its up rows are 2x unit vectors and its
    FC2 is the identity, so y_n = w * silu(x_n) * 2 x_n; expert 0 (gate 1x, up 1x) adds
    w' * silu(x_n) * x_n.  Scales are 1 (exact in fp16), X is exact in fp16."""
    b1, b2 = bits
    H = I = 32
    bs = 32
    E = 3
    x = np.linspace(-3, 3, H).round(3)
    X = wl.cast(x.reshape(1, H), "f16")
    xv = X.view(np.float16).astype(np.float64)[0]
    gate_row = (lambda i: 2 * i) if layout == "interleaved" else (lambda i: i)
    up_row = (lambda i: 2 * i + 1) if layout == "interleaved" else (lambda i: I + i)
    fc1 = np.zeros((E, 2 * I, oracle.row_bytes(H, b1, bs)), np.uint8)
    fc2 = np.zeros((E, H, oracle.row_bytes(I, b2, bs)), np.uint8)
    for e, up_val in ((0, 1), (1, 2), (2, 3)):
        gcols = [None] * (2 * I)
        for i in range(I):
            gcols[gate_row(i)] = i
        fc1[e] = _unit_rows(2 * I, H, b1, bs, gcols, 1)
        ucodes = oracle.unpack_codes(fc1[e], 2 * I, H, b1, bs)
        for i in range(I):
            ucodes[up_row(i)] = 1 << (b1 - 1)
            ucodes[up_row(i), i] += up_val
        fc1[e] = oracle.pack_codes(ucodes, b1, bs)
        fc2[e] = _unit_rows(H, I, b2, bs, list(range(H)), 1)
    s1 = wl.cast(np.ones((E, 2 * I, 1)), "f16")
    s2 = wl.cast(np.ones((E, H, 1)), "f16")
    d = np.float32(math.log(3.0))
    logits = np.array([[d, 0.0, -4.0]], np.float32)  # experts 0 and 1 selected, weights 3/4, 1/4
    Y = oracle.qmoe(X, "f16", logits, 2, True, fc1, s1, None, b1, fc2, s2, None, b2, I, bs, layout)
    e = math.exp(float(d))
    w0, w1 = e / (e + 1), 1 / (e + 1)
    silu = xv / (1 + np.exp(-xv))
    ref = w0 * silu * xv + w1 * silu * 2 * xv
    assert np.allclose(Y[0], ref, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
def test_qmoe_single_expert_is_two_matmuls(layout):
    g = wl.rng(14)
    T, H, I, bs = 3, 64, 64, 32
    d = wl.moe_layer(g, T, H, I, 1, 3, 4, bs, "bf16", with_zp=True)
    Y = oracle.qmoe(d["X"], "bf16", d["logits"], 1, True, d["fc1_w"], d["fc1_scales"], d["fc1_zp"],
                    3, d["fc2_w"], d["fc2_scales"], d["fc2_zp"], 4, I, bs, layout)
    GU = oracle.mnb_matmul(d["X"], "bf16", d["fc1_w"][0], d["fc1_scales"][0], "bf16", d["fc1_zp"][0],
                           2 * I, H, 3, bs)
    gate = GU[:, 0::2] if layout == "interleaved" else GU[:, :I]
    up = GU[:, 1::2] if layout == "interleaved" else GU[:, I:]
    h = gate / (1 + np.exp(-gate)) * up
    W2 = oracle.dequantize(d["fc2_w"][0], d["fc2_scales"][0], "bf16", d["fc2_zp"][0], H, I, 4, bs)
    assert np.allclose(Y, h @ W2.T, rtol=1e-12, atol=1e-12)


def test_qmoe_token_subset_and_fc2_scale_doubling():
    g = wl.rng(15)
    T, H, I, E, bs = 5, 64, 32, 6, 32
    d = wl.moe_layer(g, T, H, I, E, 4, 3, bs, "f16", skew=True)
    args = lambda s2: (d["X"], "f16", d["logits"], 3, True, d["fc1_w"], d["fc1_scales"], None, 4,
                       d["fc2_w"], s2, None, 3, I, bs)
    full = oracle.qmoe(*args(d["fc2_scales"]), threads=2)
    sub = oracle.qmoe(*args(d["fc2_scales"]), tokens=[4, 1])
    assert np.array_equal(sub, full[[4, 1]])
    s2x = wl.cast(d["fc2_scales"].view(np.float16).astype(np.float32) * 2, "f16")
    assert np.array_equal(oracle.qmoe(*args(s2x)), 2 * full)


def test_qmoe_unnormalised_weights_are_softmax_probabilities():
    g = wl.rng(16)
    T, H, I, E, bs = 2, 32, 32, 4, 32
    d = wl.moe_layer(g, T, H, I, E, 4, 4, bs, "f16")
    one = lambda k, norm: oracle.qmoe(d["X"], "f16", d["logits"], k, norm, d["fc1_w"], d["fc1_scales"],
                                      None, 4, d["fc2_w"], d["fc2_scales"], None, 4, I, bs)
    # with k = E and no renormalisation the weights are the full softmax, which sums to one,
    # so the result equals the renormalised one up to rounding
    assert np.allclose(one(E, False), one(E, True), rtol=1e-13, atol=1e-13)


# ------------------------------------------- QMoE optional inputs (biases, aggregation)

def _zero_weight_layer(g, E, H, I, bits, bs, act):
    """Experts whose dequantised weights are all zero (unit scales, every code equal to
    the implicit zero point): each projection is its bias alone."""
    z = 1 << (bits - 1)
    fc1 = np.stack([oracle.pack_codes(np.full((2 * I, H), z, np.uint8), bits, bs) for _ in range(E)])
    fc2 = np.stack([oracle.pack_codes(np.full((H, I), z, np.uint8), bits, bs) for _ in range(E)])
    s1 = wl.cast(np.ones((E, 2 * I, H // bs)), act)
    s2 = wl.cast(np.ones((E, H, I // bs)), act)
    return fc1, s1, fc2, s2


def _topk_softmax(logits, k):
    """Top-k by value, ties to the lower index (a stable sort of -logit), weights
    renormalised over the selected probabilities."""
    idx = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits.astype(np.float64), idx, axis=1)
    p = np.exp(sel - sel[:, :1])
    return idx, p / p.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("with_agg", [False, True])
def test_qmoe_fc2_bias_and_aggregation_weights_closed_form(with_agg):
    """All weights zero: FC1 gives its bias alone, FC2 gives its bias alone, so
    Y[t] = sum_j c_j fc2_bias[e_j], c_j the routing weight of slot j, or with
    aggregation weights c_j = agg[t, e_j] (the selection still follows the logits)."""
    g = wl.rng(21)
    T, H, I, E, k, bs, bits = 4, 64, 32, 6, 3, 32, 4
    fc1, s1, fc2, s2 = _zero_weight_layer(g, E, H, I, bits, bs, "f16")
    X = wl.normal(g, (T, H), "f16")
    logits = wl.router_logits(g, T, E)
    b1 = wl.normal(g, (E, 2 * I), "f16")
    b2 = wl.normal(g, (E, H), "f16")
    agg = wl.uniform(g, (T, E), 0.0, 1.0) if with_agg else None
    Y = oracle.qmoe_ex(X, "f16", logits, "f32", k, True, fc1, s1, None, b1, bits, fc2, s2, None, b2, bits, I, bs,
                       agg=agg)
    idx, w = _topk_softmax(logits, k)
    if with_agg:
        w = np.take_along_axis(agg.astype(np.float64), idx, axis=1)
    b2v = b2.view(np.float16).astype(np.float64)
    ref = np.einsum("tj,tjh->th", w, b2v[idx])
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
def test_qmoe_fc1_bias_closed_form(layout):
    """FC1 weights zero, FC2 the identity (H = I, explicit zero point 0, codes 1 on the
    diagonal, unit scales): Y[t, n] = sum_j w_j silu(bg[e_j, n]) bu[e_j, n] with bg and bu
    the FC1 bias entries of gate and up rows of pair n in the layout's row order."""
    g = wl.rng(22)
    T, H, I, E, k, bs, bits = 3, 32, 32, 5, 2, 32, 4
    z = 1 << (bits - 1)
    fc1 = np.stack([oracle.pack_codes(np.full((2 * I, H), z, np.uint8), bits, bs) for _ in range(E)])
    eye = np.eye(H, I, dtype=np.uint8)
    fc2 = np.stack([oracle.pack_codes(eye, bits, bs) for _ in range(E)])
    z2 = np.stack([oracle.pack_zero_points(np.zeros((H, I // bs), np.uint8), bits) for _ in range(E)])
    s1 = wl.cast(np.ones((E, 2 * I, H // bs)), "bf16")
    s2 = wl.cast(np.ones((E, H, I // bs)), "bf16")
    X = wl.normal(g, (T, H), "bf16")
    logits = wl.router_logits(g, T, E)
    b1 = wl.normal(g, (E, 2 * I), "bf16")
    Y = oracle.qmoe_ex(X, "bf16", logits, "f32", k, True, fc1, s1, None, b1, bits, fc2, s2, z2, None, bits, I, bs,
                       layout)
    idx, w = _topk_softmax(logits, k)
    b = torch.from_numpy(b1.view(np.int16)).view(torch.bfloat16).double().numpy()
    bg = b[:, 0::2] if layout == "interleaved" else b[:, :I]
    bu = b[:, 1::2] if layout == "interleaved" else b[:, I:]
    h = bg / (1 + np.exp(-bg)) * bu  # [E, I]
    ref = np.einsum("tj,tjn->tn", w, h[idx])
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("ldt", ["f16", "bf16"])
def test_qmoe_half_logits_equal_their_widened_values(ldt):
    """Router logits in a 16-bit type select and weigh exactly like fp32 logits that
    hold the widened values."""
    g = wl.rng(23)
    T, H, I, E, k, bs = 3, 64, 32, 8, 3, 32
    d = wl.moe_layer(g, T, H, I, E, 4, 3, bs, "f16")
    lh = wl.cast(np.round(d["logits"] * 4) / 4, ldt)  # coarse values: ties in the selection too
    lf = as_f64(lh, ldt).astype(np.float32).reshape(T, E)
    args = lambda L, dt: oracle.qmoe_ex(d["X"], "f16", L, dt, k, True, d["fc1_w"], d["fc1_scales"], None, None, 4,
                                        d["fc2_w"], d["fc2_scales"], None, None, 3, I, bs)
    assert np.array_equal(args(lh.reshape(T, E), ldt), args(lf, "f32"))


def test_qmoe_ex_without_options_is_qmoe():
    g = wl.rng(24)
    T, H, I, E, k, bs = 2, 64, 64, 4, 2, 64
    d = wl.moe_layer(g, T, H, I, E, 3, 3, bs, "bf16", with_zp=True)
    a = oracle.qmoe(d["X"], "bf16", d["logits"], k, False, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], 3, d["fc2_w"],
                    d["fc2_scales"], d["fc2_zp"], 3, I, bs)
    b = oracle.qmoe_ex(d["X"], "bf16", d["logits"], "f32", k, False, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], None,
                       3, d["fc2_w"], d["fc2_scales"], d["fc2_zp"], None, 3, I, bs)
    assert np.array_equal(a, b)


# ------------------------------------------------- INT3 quantizer (producer)
# The symmetric grouped INT3 round-to-nearest policy quoted in "INT3 QMoE CUDA
# correctness baseline and Qwen experimental results" (Olive producer summary).

def _f16_bits(x32):
    with np.errstate(over="ignore"):  # values past 65504 become infinity, as they should
        return np.asarray(x32, np.float32).astype(np.float16).view(np.uint16)


def _bf16_bits(x32):
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_int3_worked_example():
    """max|w| = 3.5 gives scale 1: codes are round(w) + 4 with ties to even, +3.5
    saturating at 7 and -3.5 landing on 0."""
    w = np.zeros((1, 32), np.float32)
    w[0, :8] = [3.5, -3.5, 1.0, 1.5, 2.5, -0.5, 0.0, -2.5]
    packed, scales, bad = oracle.quantize_int3(w, "f32", 32, "f16")
    assert not bad.any() and scales[0, 0] == 0x3C00  # binary16 1.0
    codes = oracle.unpack_codes(packed, 1, 32, 3, 32)[0]
    assert list(codes[:8]) == [7, 0, 5, 6, 6, 4, 4, 2]
    assert (codes[8:] == 4).all()


def test_quantize_int3_all_zero_block_stores_one_over_three_and_a_half():
    w = np.zeros((2, 64), np.float32)
    w[1, 40] = 1.0  # second row: the first block is zero, the second is not
    for s_dtype, bits_of in (("f16", _f16_bits), ("bf16", _bf16_bits)):
        packed, scales, bad = oracle.quantize_int3(w, "f32", 32, s_dtype)
        assert not bad.any()
        one_over = bits_of(np.float32(1.0) / np.float32(3.5))
        assert scales[0, 0] == one_over and scales[0, 1] == one_over and scales[1, 0] == one_over
        assert scales[1, 1] == bits_of(np.float32(1.0) / np.float32(3.5))  # max|w| = 1 as well
        codes = oracle.unpack_codes(packed, 2, 64, 3, 32)
        assert (codes[0] == 4).all() and (codes[1, :32] == 4).all()
        assert codes[1, 40] == 7  # 1 / (1/3.5) = 3.5 saturates


@pytest.mark.parametrize("s_dtype", ["f16", "bf16"])
def test_quantize_int3_stored_scale_rounding_matches_library_casts(s_dtype):
    """Per-block scales over many magnitudes (subnormal, normal, overflowing
    binary16) equal numpy's / torch's round-to-nearest-even casts of the binary32
    quotient max|w| / 3.5."""
    g = np.random.default_rng(31)
    N, bs = 400, 32
    mag = np.float32(10.0) ** g.uniform(-9, 6, size=N).astype(np.float32)
    w = (g.standard_normal((N, bs)).astype(np.float32) * mag[:, None]).astype(np.float32)
    packed, scales, bad = oracle.quantize_int3(w, "f32", bs, s_dtype)
    q = np.abs(w).max(axis=1).astype(np.float32) / np.float32(3.5)
    ref = _f16_bits(q) if s_dtype == "f16" else _bf16_bits(q)
    assert np.array_equal(scales[:, 0], ref)
    stored = (ref.view(np.float16).astype(np.float64) if s_dtype == "f16" else as_f64(ref, "bf16"))
    assert np.array_equal(bad[:, 0], ~np.isfinite(stored) | (stored == 0))
    if s_dtype == "f16":
        assert (stored[~bad[:, 0]] < 2.0 ** -14).any() and bad[:, 0].any()  # subnormals kept, some rejected


@pytest.mark.parametrize("s_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [32, 64, 128])
def test_quantize_int3_codes_are_the_nearest_levels(s_dtype, bs):
    """Every code picks, among the eight levels (q - 4) * scale, the one nearest
    to w in units of the binary32 quotient w / scale; an exact half goes to the
    even level; the reconstruction error is at most half a scale step except at
    the saturated top."""
    g = np.random.default_rng(bs * 7 + len(s_dtype))
    N, K = 9, 4 * bs
    w = g.standard_normal((N, K)).astype(np.float32)
    packed, scales, bad = oracle.quantize_int3(w, "f32", bs, s_dtype)
    assert not bad.any()
    codes = oracle.unpack_codes(packed, N, K, 3, bs).astype(np.int64)
    s = scales.astype(np.float64) if s_dtype == "f32" else (
        scales.view(np.float16).astype(np.float64) if s_dtype == "f16" else as_f64(scales, "bf16"))
    s32 = np.repeat(s, bs, axis=1).astype(np.float32)
    r = (w / s32).astype(np.float64)
    levels = np.arange(-4, 4, dtype=np.float64)
    dist = np.abs(r[..., None] - levels)
    best = dist.min(axis=-1)
    chosen = dist[np.arange(N)[:, None], np.arange(K)[None, :], codes]
    assert np.array_equal(chosen, best)
    ties = (dist == best[..., None]).sum(axis=-1) > 1
    assert ((codes[ties] - 4) % 2 == 0).all()
    err = np.abs(w - np.repeat(s, bs, axis=1) * (codes - 4))
    top = codes == 7
    assert (err[~top] <= 0.5 * np.repeat(s, bs, axis=1)[~top] * (1 + 1e-6)).all()


def test_quantize_int3_rejects_non_finite_and_zero_rounded_blocks():
    w = np.ones((4, 64), np.float32)
    w[0, 3] = np.nan
    w[1, 40] = np.inf
    w[2, :32] = 1e-9  # binary16 scale 2.9e-10 rounds to zero
    w[3, :32] = 3.5e-6  # scale 1e-6: a binary16 subnormal, kept
    packed, scales, bad = oracle.quantize_int3(w, "f32", 32, "f16")
    assert bad.tolist() == [[True, False], [False, True], [True, False], [False, False]]
    assert scales[3, 0] < 0x0400  # subnormal binary16 pattern
    codes = oracle.unpack_codes(packed, 4, 64, 3, 32)
    assert (codes[0, :32] == 4).all() and (codes[2, :32] == 4).all()
    # the same tiny block is representable with a bfloat16 scale
    _, _, bad_bf = oracle.quantize_int3(w[2:3], "f32", 32, "bf16")
    assert not bad_bf.any()


@pytest.mark.parametrize("w_dtype", ["f16", "bf16"])
def test_quantize_int3_half_inputs_equal_their_binary32_values(w_dtype):
    g = np.random.default_rng(5)
    w16 = wl.normal(g, (5, 128), w_dtype)
    a = oracle.quantize_int3(w16, w_dtype, 64, "f16")
    b = oracle.quantize_int3(as_f64(w16, w_dtype).astype(np.float32).reshape(5, 128), "f32", 64, "f16")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _boundary_cases(patterns_f64):
    """Every midpoint between adjacent representable values and its binary32
    neighbours one ulp below and above, plus the values themselves."""
    v = np.sort(np.unique(patterns_f64[np.isfinite(patterns_f64)]))
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    xs = np.concatenate([v.astype(np.float32), mids, np.nextafter(mids, np.float32(-np.inf)),
                         np.nextafter(mids, np.float32(np.inf))])
    return xs[np.isfinite(xs)]


def test_half_rounding_at_every_boundary_matches_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xs = _boundary_cases(pats.view(np.float16).astype(np.float64))
    xs = np.concatenate([xs, np.float32([65519.996, 65520.0, 65536.0, 1e30, -1e30, np.inf, -np.inf])])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_to_half_bits(xs, "f16"), ref)


def test_bfloat16_rounding_at_every_boundary_matches_torch():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xs = _boundary_cases(as_f64(pats, "bf16"))
    xs = np.concatenate([xs, np.float32([3.4e38, -3.4e38, np.inf, -np.inf])])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_to_half_bits(xs, "bf16"), ref)


# ---------------------------------------------------------------- prepacked layout

PREPACK_HEADER = struct.Struct("<IIqqiiiiqqqqQ")


def _lsb_first_codes(row: np.ndarray, n: int, bits: int) -> list[int]:
    """Codes 0 .. n-1 of a row-local LSB-first stream, bit by bit."""
    bitv = np.unpackbits(row, bitorder="little")
    return [int(sum(int(bitv[bits * j + t]) << t for t in range(bits))) for j in range(n)]


def _decode_prepacked_chunk(ch: bytes, bits: int) -> list[int]:
    """The 32 codes of one prepacked chunk, read back from the layout's definition."""
    if bits == 4:
        return [(ch[j // 2] >> (4 * (j % 2))) & 15 for j in range(32)]
    q = [0] * 32
    for g in range(3):
        for b in range(4):
            byte = ch[4 * g + b]
            q[8 * g + 2 * b] = byte & 7
            q[8 * g + 2 * b + 1] = (byte >> 3) & 7
    for b in range(4):
        q[24 + 2 * b] = (ch[b] >> 6) | (((ch[8 + b] >> 6) & 1) << 2)
        q[25 + 2 * b] = (ch[4 + b] >> 6) | (((ch[8 + b] >> 7) & 1) << 2)
    return q


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("s_dtype,with_zp", [("f32", False), ("f16", True), ("bf16", True)])
def test_prepack_decodes_back_to_the_row_local_weight(bits, bs, s_dtype, with_zp):
    """The oracle's prepacked bytes, decoded field by field from the layout's
    definition: header values, every stored code (padding codes included), the
    scale and zero-point bytes, zero padding, rows of whole 16-byte units."""
    N, K = 5, 200
    g = wl.rng(0xB0 + bits + bs)
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, s_dtype, with_zp)
    out = oracle.prepack(packed, scales, s_dtype, zp, N, K, bits, bs, identity=0x1234_5678_9ABC_DEF0)
    (magic, version, n_, k_, bits_, bs_, sdt, has_zp, stride, s_off, z_off, total,
     ident) = PREPACK_HEADER.unpack_from(out.tobytes(), 0)
    nb = -(-K // bs)
    ss = 4 if s_dtype == "f32" else 2
    zr = (nb * bits + 7) // 8
    assert (magic, version, n_, k_, bits_, bs_) == (0x50424E4D, 1, N, K, bits, bs)
    assert out[:4].tobytes() == b"MNBP"
    assert (sdt, has_zp, ident) == (oracle.DTYPES[s_dtype], int(with_zp), 0x1234_5678_9ABC_DEF0)
    code_bytes = nb * bs * bits // 8
    raw = code_bytes + nb * ss + (zr if with_zp else 0)
    assert stride % 16 == 0 and raw <= stride < raw + 16
    assert (s_off, z_off) == (code_bytes, code_bytes + nb * ss if with_zp else -1)
    assert total == out.size == 128 + N * stride
    assert not out[PREPACK_HEADER.size:128].any()
    sb = np.ascontiguousarray(scales).view(np.uint8).reshape(N, nb * ss)
    for n in range(N):
        row = out[128 + n * stride:128 + (n + 1) * stride]
        want = _lsb_first_codes(packed[n], nb * bs, bits)
        got = []
        for c in range(nb * bs // 32):
            got += _decode_prepacked_chunk(row[c * 4 * bits:(c + 1) * 4 * bits].tobytes(), bits)
        assert got == want
        assert np.array_equal(row[s_off:s_off + nb * ss], sb[n])
        end = s_off + nb * ss
        if with_zp:
            assert np.array_equal(row[z_off:z_off + zr], zp[n])
            end = z_off + zr
        assert not row[end:].any()


def test_prepack_int3_chunk_worked_example():
    """Codes c_j = j mod 8 in one chunk: the regrouped words worked out by hand from
    the layout (bytes of W0: 8, 26, 44, 62 plus the low bits of c_24, c_26, c_28,
    c_30 = 0, 2, 4, 6 in bits 6-7; W2 carries their third bits)."""
    codes = np.array([[j % 8 for j in range(32)]], np.uint8)
    packed = oracle.pack_codes(codes, 3, 32)
    out = oracle.prepack(packed, np.ones((1, 1), np.float32), "f32", None, 1, 32, 3, 32)
    ch = list(out[128:140])
    # W0 byte b: c_{2b} | c_{2b+1} << 3 | (c_{24+2b} & 3) << 6, c_{24+2b} = 0, 2, 4, 6
    assert ch[0:4] == [0 | 1 << 3 | 0 << 6, 2 | 3 << 3 | 2 << 6, 4 | 5 << 3 | 0 << 6, 6 | 7 << 3 | 2 << 6]
    # W1 byte b: c_{8+2b} | c_{9+2b} << 3 | (c_{25+2b} & 3) << 6, c_{25+2b} = 1, 3, 5, 7
    assert ch[4:8] == [0 | 1 << 3 | 1 << 6, 2 | 3 << 3 | 3 << 6, 4 | 5 << 3 | 1 << 6, 6 | 7 << 3 | 3 << 6]
    # W2 byte b: c_{16+2b} | c_{17+2b} << 3 | bit2(c_{24+2b}) << 6 | bit2(c_{25+2b}) << 7
    assert ch[8:12] == [0 | 1 << 3 | 0 << 6 | 0 << 7, 2 | 3 << 3 | 0 << 6 | 0 << 7,
                        4 | 5 << 3 | 1 << 6 | 1 << 7, 6 | 7 << 3 | 1 << 6 | 1 << 7]
