"""GPU parity of mnb_matmul's tensor-core path (tcgen05, fp16/bf16 activations,
M >= 16) against the oracle: every output of every activation row where the
oracle's cost is at most 1e10 multiply-adds, else of at least 64 sampled rows.

Rules (tests/_util.py): fp32 outputs the fp32 rule (the path then adds the
16-bit weights' rounding remainder in a second pass); fp16 outputs the
elementwise 16-bit rule; bf16 outputs from bf16 activations the bf16
tensor-core rule, with the elementwise misses printed."""
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import assert_close, empty_guarded, guarded_workspace, guards_intact, to_dev, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1


def seed(*key):
    return zlib.crc32(repr(key).encode())


def run(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, y_dt):
    A_d = to_dev(A, a_dt)
    M = A_d.numel() // K
    Y, full = empty_guarded(M * N, y_dt)
    mnb.mnb_matmul(A_d, to_dev(packed), to_dev(scales, s_dt), None if zp is None else to_dev(zp), N, bits, bs, Y,
                   K=K, M=M)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(M, N)


def sample_rows(M, N, K, n=64):
    """Every row where the oracle's cost M*N*K is at most 1e10 multiply-adds,
    else the first, middle and last rows plus distinct random ones, >= n rows."""
    if M * N * K <= 1e10 or M <= n:
        return list(range(M))
    g = wl.rng(M)
    rows = {0, M // 2, M - 1}
    while len(rows) < n:
        rows.add(int(g.integers(0, M)))
    return sorted(rows)


def check(M, K, N, bits, bs, a_dt="bf16", s_dt="f32", y_dt="bf16", with_zp=False, key=()):
    g = wl.rng(seed(M, K, N, bits, bs, a_dt, s_dt, y_dt, with_zp, *key))
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, s_dt, with_zp)
    A = wl.normal(g, (M, K), a_dt)
    y = run(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, y_dt)
    rows = sample_rows(M, N, K)
    ref = oracle.mnb_matmul(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, mrows=rows, threads=THREADS)
    assert_close(y[rows], ref, y_dt, a_dt, tensor_cores=M >= 16,
                 label=f"M={M} K={K} N={N} bits={bits} bs={bs} {a_dt}/{s_dt}->{y_dt}")


@pytest.mark.parametrize("M", [16, 128, 512, 2048])
@pytest.mark.parametrize("name,K,N", wl.QWEN3_1P7B_PROJECTIONS + [wl.QWEN3_1P7B_LM_HEAD])
def test_qwen3_prefill_projection(M, name, K, N):
    """Same INT4 weights layout as the decode suite: bf16 activations, fp32 scales, bf16 out."""
    check(M, K, N, 4, 32, key=(name,))


@pytest.mark.parametrize("M,K,N,bs", [(128, 2080, 512, 32), (512, 2072, 384, 32), (128, 2080, 640, 64),
                                      (300, 2080, 256, 128), (128, 2048, 6147, 32), (512, 2048, 6147, 32)])
def test_tails(M, K, N, bs):
    check(M, K, N, 4, bs)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("N", [1, 48, 127])
def test_fewer_weight_rows_than_a_tile(bits, N):
    """N < 128: the packed-row and scale tiles of the single weight tile run past
    the matrix and read zeros there; all N outputs of the sampled rows are checked."""
    check(64, 1024, N, bits, 64, "bf16", "bf16", "bf16", with_zp=bits == 3)


@pytest.mark.parametrize("M", [8, 9, 17, 100, 255, 257, 1000])
def test_row_counts(M):
    check(M, 1024, 768, 4, 32)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("with_zp", [False, True])
def test_formats(bits, bs, with_zp):
    check(256, 2048, 1024, bits, bs, "f16", "f16", "f16", with_zp)


@pytest.mark.parametrize("a_dt,s_dt,y_dt", [("bf16", "bf16", "bf16"), ("f16", "f32", "f32"), ("bf16", "f32", "f32"),
                                            ("f16", "f16", "bf16")])
def test_dtypes(a_dt, s_dt, y_dt):
    check(200, 1536, 896, 3, 64, a_dt, s_dt, y_dt, with_zp=True)


@pytest.mark.parametrize("bits", [3, 4])
def test_integer_data_is_bit_exact(bits):
    """scales = 1, zero points 0, integer activations: the bf16 tile holds the codes
    exactly and every fp32 partial sum is an integer below 2^24."""
    g = wl.rng(seed("tc-int", bits))
    M, N, K, bs = 200, 384, 2048, 64
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    zp = oracle.pack_zero_points(np.zeros((N, K // bs), np.uint8), bits)
    Af = g.integers(-4, 5, size=(M, K)).astype(np.float32)
    y = run(wl.cast(Af, "bf16"), "bf16", packed, np.ones((N, K // bs), np.float32), "f32", zp, N, K, bits, bs, "f32")
    assert np.array_equal(y, (Af.astype(np.int64) @ codes.astype(np.int64).T).astype(np.float64))


def test_deterministic_and_matches_across_paths():
    """M = 8 (tensor cores) against M = 4 + 4 (CUDA cores) on the same rows."""
    g = wl.rng(seed("paths"))
    K, N = 2048, 1024
    packed, scales, _ = wl.quantized_weight(g, N, K, 4, 32)
    A = wl.normal(g, (8, K), "bf16")
    y8 = run(A, "bf16", packed, scales, "f32", None, N, K, 4, 32, "f32")
    y8b = run(A, "bf16", packed, scales, "f32", None, N, K, 4, 32, "f32")
    assert np.array_equal(y8, y8b)
    y4 = np.concatenate([run(A[:4], "bf16", packed, scales, "f32", None, N, K, 4, 32, "f32"),
                         run(A[4:], "bf16", packed, scales, "f32", None, N, K, 4, 32, "f32")])
    assert np.max(np.abs(y8 - y4)) <= 2e-2 * np.sqrt(np.mean(y4 ** 2))


@pytest.mark.parametrize("bits,bs", [(4, 32), (3, 64)])
@pytest.mark.parametrize("a_dt", ["bf16", "f16"])
def test_fp32_output_carries_the_weights_rounding_remainder(bits, bs, a_dt):
    """An fp32 output from 16-bit activations: the tensor cores take the dequantised
    weight rounded to the activation's 16-bit type, then a second pass adds the
    product with the remainder s (q - z) - round16(s (q - z)), itself rounded to
    16 bits.  The result meets the fp32 rule and sits far closer to the exact
    product than a product of 16-bit-rounded weights does."""
    g = wl.rng(seed("remainder", bits, bs, a_dt))
    M, K, N = 64, 2048, 512
    packed, scales, _ = wl.quantized_weight(g, N, K, bits, bs)
    A = wl.normal(g, (M, K), a_dt)
    y = run(A, a_dt, packed, scales, "f32", None, N, K, bits, bs, "f32")
    W = oracle.dequantize(packed, scales, "f32", None, N, K, bits, bs)
    tdt = torch.bfloat16 if a_dt == "bf16" else torch.float16
    Af = torch.from_numpy(A.view(np.int16)).view(tdt).double().numpy()
    exact = oracle.mnb_matmul(A, a_dt, packed, scales, "f32", None, N, K, bits, bs, threads=THREADS)
    one_pass = Af @ torch.from_numpy(W.astype(np.float32)).to(tdt).double().numpy().T
    rel = lambda d: float(np.sqrt(np.mean(d * d)) / np.sqrt(np.mean(exact * exact)))
    assert_close(y, exact, "f32")
    assert rel(y - exact) <= 0.05 * rel(one_pass - exact)


@pytest.mark.parametrize("M,K,N,bits,bs", [(16, 2048, 4096, 4, 32), (16, 6144, 2048, 4, 32), (32, 2080, 2048, 3, 32),
                                           (64, 2048, 1024, 3, 64), (24, 2304, 640, 4, 128)])
def test_split_k_against_unsplit(M, K, N, bits, bs):
    """Output tiles too few to fill the GPU: K is split across CTAs (fp32 partial sums in
    the workspace, then a reduction; an fp32 output runs the remainder pass the same
    way).  Checked against the oracle, and against the same call with no workspace
    (no split): equal up to the order of the fp32 additions."""
    g = wl.rng(seed("splitk", M, K, N, bits, bs))
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, "bf16", bits == 3)
    A = wl.normal(g, (M, K), "bf16")
    need = mnb.mnb_matmul_workspace_size(M, K, N, bits, bs, mnb.BF16)
    assert need > 0, "these shapes leave SMs idle without a split"
    A_d, B_d, S_d = to_dev(A, "bf16"), to_dev(packed), to_dev(scales, "bf16")
    Z_d = None if zp is None else to_dev(zp)
    ys = []
    for nbytes in (need, 0):
        ws, ws_full = guarded_workspace(nbytes)
        Y, full = empty_guarded(M * N, "f32")
        mnb.mnb_matmul(A_d, B_d, S_d, Z_d, N, bits, bs, Y, ws, K=K, M=M)  # 0 bytes: no split
        torch.cuda.synchronize()
        assert guards_intact(full), "write outside Y"
        assert guards_intact(ws_full, 256), "write outside the split-K workspace"
        assert mnb.mnb_get_last_device_error() == 0
        ys.append(to_f64(Y).reshape(M, N))
    ref = oracle.mnb_matmul(A, "bf16", packed, scales, "bf16", zp, N, K, bits, bs, threads=THREADS)
    assert_close(ys[0], ref, "f32")
    assert_close(ys[1], ref, "f32")
    rel = np.max(np.abs(ys[0] - ys[1])) / max(np.max(np.abs(ys[1])), 1e-30)
    assert rel <= 1e-5, rel
