"""GPU parity of mnb_matmul's SIMT path (M = 1 decode GEMV and small M)
against the oracle, through the C ABI."""
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import (CODE, assert_close, assert_f32_close, empty_guarded, f32_error, guards_intact, to_dev,
                         to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1


def seed(*key):
    return zlib.crc32(repr(key).encode())


def run(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, y_dt="f32", M=None):
    A_d = to_dev(A, a_dt)
    M = A_d.numel() // K if M is None else M
    Y, full = empty_guarded(M * N, y_dt)
    mnb.mnb_matmul(A_d, to_dev(packed), to_dev(scales, s_dt), None if zp is None else to_dev(zp), N, bits, bs, Y,
                   K=K, M=M)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(M, N)


def case(g, M, K, N, bits, bs, a_dt="f32", s_dt="f32", with_zp=False):
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, s_dt, with_zp)
    A = wl.normal(g, (M, K), a_dt)
    return A, packed, scales, zp


def test_tiny_case():
    t = wl.TINY
    g = wl.rng(0)
    A, packed, scales, zp = case(g, t["M"], t["K"], t["N"], t["bits"], t["bs"])
    y = run(A, "f32", packed, scales, "f32", None, t["N"], t["K"], 4, 32)
    ref = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, t["N"], t["K"], 4, 32)
    assert_f32_close(y, ref)


@pytest.mark.parametrize("name,K,N", wl.QWEN3_1P7B_PROJECTIONS + [wl.QWEN3_1P7B_LM_HEAD])
def test_qwen3_decode_projection(name, K, N):
    g = wl.rng(seed("decode", name))
    A, packed, scales, _ = case(g, 1, K, N, 4, 32)
    y = run(A, "f32", packed, scales, "f32", None, N, K, 4, 32)
    ref = oracle.mnb_matmul(A, "f32", packed, scales, "f32", None, N, K, 4, 32, threads=THREADS)
    # the margin of the float-image dequantisation (sums of pre-scaled activations
    # cancel before the block scale is applied) against the 1e-3 rule
    print(f"[decode {name} K={K} N={N}] fp32 relative error {f32_error(y, ref):.3g} (rule 1e-3)")
    assert_f32_close(y, ref)
    if name == "qkv":  # the fused QKV output splits by column offset [2048, 1024, 1024]
        o = 0
        for w in wl.QKV_SPLIT:
            assert_f32_close(y[:, o:o + w], ref[:, o:o + w])
            o += w


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("with_zp", [False, True])
def test_formats(bits, bs, with_zp):
    g = wl.rng(seed("formats", bits, bs, with_zp))
    K, N = 2048, 1000
    A, packed, scales, zp = case(g, 1, K, N, bits, bs, with_zp=with_zp)
    y = run(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    assert_f32_close(y, oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs, threads=THREADS))


@pytest.mark.parametrize("a_dt,s_dt,y_dt", [("f16", "f16", "f16"), ("bf16", "bf16", "bf16"), ("bf16", "f32", "bf16"),
                                            ("f16", "f32", "f32"), ("bf16", "bf16", "f32"), ("f32", "f32", "bf16")])
@pytest.mark.parametrize("bits", [3, 4])
def test_dtypes(a_dt, s_dt, y_dt, bits):
    g = wl.rng(seed("dtypes", a_dt, s_dt, y_dt, bits))
    K, N, bs = 1536, 777, 64
    A, packed, scales, zp = case(g, 1, K, N, bits, bs, a_dt, s_dt, with_zp=True)
    y = run(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, y_dt)
    assert_close(y, oracle.mnb_matmul(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, threads=THREADS), y_dt)


@pytest.mark.parametrize("K,N,bs,bits", [(2080, 512, 32, 4), (2072, 512, 32, 4), (2080, 512, 64, 4), (2080, 512, 128, 4),
                                         (2048, 6147, 32, 4), (2072, 300, 32, 3), (2080, 129, 64, 3), (33, 5, 32, 4),
                                         (1, 1, 32, 4), (1, 3, 128, 3), (256, 127, 32, 3), (6144, 1, 32, 4)])
def test_tails(K, N, bs, bits):
    g = wl.rng(seed("tails", K, N, bs, bits))
    A, packed, scales, zp = case(g, 1, K, N, bits, bs, with_zp=(N % 2 == 1))
    y = run(A, "f32", packed, scales, "f32", zp, N, K, bits, bs)
    assert_f32_close(y, oracle.mnb_matmul(A, "f32", packed, scales, "f32", zp, N, K, bits, bs, threads=THREADS))


@pytest.mark.parametrize("M", [2, 3, 4, 5, 16])
@pytest.mark.parametrize("a_dt", ["f32", "bf16"])
def test_small_m(M, a_dt):
    g = wl.rng(seed("smallm", M, a_dt))
    K, N, bs = 2048, 1024, 32
    y_dt = "f32" if a_dt == "f32" else "bf16"
    A, packed, scales, zp = case(g, M, K, N, 4, bs, a_dt)
    y = run(A, a_dt, packed, scales, "f32", None, N, K, 4, bs, y_dt)
    assert_close(y, oracle.mnb_matmul(A, a_dt, packed, scales, "f32", None, N, K, 4, bs, threads=THREADS), y_dt,
                 a_dt, tensor_cores=M >= 16 and a_dt != "f32", label=f"small M={M}")


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("a_dt", ["f32", "f16", "bf16"])
def test_integer_data_is_bit_exact(bits, a_dt):
    """scales = 1, zero points 0, integer activations in [-4, 4]: every partial sum is an
    integer below 2^24, so an fp32 output must equal the exact result."""
    g = wl.rng(seed("intexact", bits, a_dt))
    N, K, bs, M = 300, 2048, 64, 1
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    nb = K // bs
    zp = oracle.pack_zero_points(np.zeros((N, nb), np.uint8), bits)
    Af = g.integers(-4, 5, size=(M, K)).astype(np.float32)
    A = wl.cast(Af, a_dt)
    scales = wl.cast(np.ones((N, nb), np.float32), a_dt if a_dt != "f32" else "f32")
    y = run(A, a_dt, packed, scales, a_dt, zp, N, K, bits, bs, "f32")
    exact = (Af.astype(np.int64) @ codes.astype(np.int64).T).astype(np.float64)
    assert np.array_equal(y, exact)
    assert np.array_equal(y, oracle.mnb_matmul(A, a_dt, packed, scales, a_dt, zp, N, K, bits, bs))


@pytest.mark.parametrize("bits", [3, 4])
def test_integer_data_half_output_small_k(bits):
    g = wl.rng(seed("intexact-half", bits))
    N, K, bs = 64, 16, 32
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    zp = oracle.pack_zero_points(np.zeros((N, 1), np.uint8), bits)
    Af = g.integers(-4, 5, size=(1, K)).astype(np.float32)
    for dt in ("f16", "bf16"):
        y = run(wl.cast(Af, dt), dt, packed, wl.cast(np.ones((N, 1)), dt), dt, zp, N, K, bits, bs, dt)
        assert np.array_equal(y, (Af.astype(np.int64) @ codes.astype(np.int64).T).astype(np.float64))


def test_scale_doubling_and_implicit_zero_point_are_exact():
    g = wl.rng(seed("invariants"))
    K, N = 2048, 2048
    for bits in (3, 4):
        A, packed, scales, _ = case(g, 1, K, N, bits, 32)
        y1 = run(A, "f32", packed, scales, "f32", None, N, K, bits, 32)
        y2 = run(A, "f32", packed, scales * np.float32(2), "f32", None, N, K, bits, 32)
        assert np.array_equal(y2, 2 * y1)
        zp = oracle.pack_zero_points(np.full((N, K // 32), 1 << (bits - 1), np.uint8), bits)
        y3 = run(A, "f32", packed, scales, "f32", zp, N, K, bits, 32)
        assert np.array_equal(y3, y1)


def test_repeated_calls_are_deterministic():
    g = wl.rng(seed("determinism"))
    K, N = 6144, 2048
    A, packed, scales, _ = case(g, 1, K, N, 4, 32)
    ys = [run(A, "f32", packed, scales, "f32", None, N, K, 4, 32) for _ in range(3)]
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


def test_non_canonical_padding_is_ignored():
    """A partial last block whose padding codes are random must give the same
    result as the same weights with zero padding."""
    g = wl.rng(seed("padding"))
    K, N, bs = 2072, 256, 32
    codes = g.integers(0, 16, size=(N, K), dtype=np.uint8)
    canon = oracle.pack_codes(codes, 4, bs)
    noisy = canon.copy()
    tail = oracle.row_bytes(K, 4, bs) - (K * 4) // 8
    noisy[:, -tail:] |= g.integers(0, 256, size=(N, tail), dtype=np.uint8)
    scales = wl.uniform(g, (N, oracle.n_blocks(K, bs)), 0.005, 0.02)
    A = wl.normal(g, (1, K))
    assert np.array_equal(run(A, "f32", canon, scales, "f32", None, N, K, 4, bs),
                          run(A, "f32", noisy, scales, "f32", None, N, K, 4, bs))


# ------------------------------------------- int8 activation compute (accuracy_level=4)

def run_int8a(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, y_dt="f32"):
    A_d = to_dev(A, a_dt)
    M = A_d.numel() // K
    Y, full = empty_guarded(M * N, y_dt)
    mnb.mnb_matmul_int8a(A_d, to_dev(packed), to_dev(scales, s_dt), None if zp is None else to_dev(zp), N, bits, bs, Y,
                         K=K, M=M)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(M, N)


@pytest.mark.parametrize("name,K,N", wl.QWEN3_1P7B_PROJECTIONS)
def test_int8a_decode_projection(name, K, N):
    g = wl.rng(seed("int8a", name))
    A, packed, scales, _ = case(g, 1, K, N, 4, 32)
    y = run_int8a(A, "f32", packed, scales, "f32", None, N, K, 4, 32)
    assert_f32_close(y, oracle.mnb_matmul_int8a(A, "f32", packed, scales, "f32", None, N, K, 4, 32, threads=THREADS))


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("a_dt,M", [("f16", 1), ("bf16", 3), ("f32", 16), ("bf16", 33)])
def test_int8a_formats_and_rows(bits, bs, a_dt, M):
    """Every width and block size, 16-bit and fp32 activations, M up to 33 (the mode
    runs on CUDA cores for any M), zero points, a partial last block."""
    g = wl.rng(seed("int8a-fmt", bits, bs, a_dt, M))
    K, N = 1000, 300
    A, packed, scales, zp = case(g, M, K, N, bits, bs, a_dt, "f32", with_zp=True)
    y = run_int8a(A, a_dt, packed, scales, "f32", zp, N, K, bits, bs)
    assert_f32_close(y, oracle.mnb_matmul_int8a(A, a_dt, packed, scales, "f32", zp, N, K, bits, bs, threads=THREADS))


@pytest.mark.parametrize("bits", [3, 4])
def test_int8a_integer_data_is_bit_exact(bits):
    """Integer activations whose every block reaches 127 quantise to themselves; with unit
    scales and zero points 0 every partial sum is an integer below 2^24."""
    g = wl.rng(seed("int8a-exact", bits))
    N, K, bs, M = 200, 2048, 64, 2
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    zp = oracle.pack_zero_points(np.zeros((N, K // bs), np.uint8), bits)
    Af = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    Af[:, ::bs] = 127.0
    y = run_int8a(Af, "f32", packed, np.ones((N, K // bs), np.float32), "f32", zp, N, K, bits, bs)
    assert np.array_equal(y, (Af.astype(np.int64) @ codes.astype(np.int64).T).astype(np.float64))


# ---------------------------------------- widths beyond 3 and 4 (row-local LSB-first)

@pytest.mark.parametrize("bits", [1, 2, 5, 6, 7, 8])
@pytest.mark.parametrize("bs,with_zp,a_dt,M", [(32, False, "f32", 1), (64, True, "bf16", 3), (128, True, "f16", 20)])
def test_other_widths(bits, bs, with_zp, a_dt, M):
    """mnb_matmul at widths 1, 2, 5..8 (the CUDA-core path for any M; M = 20 with 16-bit
    activations would take the tensor cores at widths 3 and 4)."""
    g = wl.rng(seed("widths", bits, bs, with_zp, a_dt, M))
    K, N = 1000, 257
    A, packed, scales, zp = case(g, M, K, N, bits, bs, a_dt, "f32", with_zp=with_zp)
    y = run(A, a_dt, packed, scales, "f32", zp, N, K, bits, bs)
    assert_f32_close(y, oracle.mnb_matmul(A, a_dt, packed, scales, "f32", zp, N, K, bits, bs, threads=THREADS))


@pytest.mark.parametrize("bits", [2, 8])
def test_other_widths_int8a(bits):
    g = wl.rng(seed("widths-int8a", bits))
    K, N, bs = 2048, 512, 64
    A, packed, scales, zp = case(g, 2, K, N, bits, bs, "bf16", "f32", with_zp=True)
    y = run_int8a(A, "bf16", packed, scales, "f32", zp, N, K, bits, bs)
    assert_f32_close(y, oracle.mnb_matmul_int8a(A, "bf16", packed, scales, "f32", zp, N, K, bits, bs, threads=THREADS))
