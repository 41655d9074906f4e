"""GPU parity of the version-1 prepacked layout, through the C ABI: the bytes
mnb_prepack writes against the oracle's restatement of the layout (bit-exact),
mnb_matmul_prepacked against the oracle's matmul, and the device-side header
check that refuses a buffer whose identity or shape does not match."""
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import SENTINEL, assert_close, empty_guarded, guards_intact, to_dev, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1
DT = {"f32": mnb.F32, "f16": mnb.F16, "bf16": mnb.BF16}


def seed(*key):
    return zlib.crc32(repr(key).encode())


def prepack(packed, scales, s_dt, zp, N, K, bits, bs, identity=0):
    n = mnb.mnb_prepack_size(N, K, bits, bs, DT[s_dt], zp is not None)
    dst = torch.full((n + 128,), SENTINEL, dtype=torch.uint8, device="cuda")
    inner = dst[64:64 + n]
    desc = mnb.mnb_prepack(to_dev(packed), to_dev(scales, s_dt), None if zp is None else to_dev(zp), N, K, bits, bs,
                           inner, identity, scale_dtype=DT[s_dt])
    torch.cuda.synchronize()
    h = dst.cpu().numpy()
    assert (h[:64] == SENTINEL).all() and (h[64 + n:] == SENTINEL).all(), "write outside the prepacked buffer"
    return desc, inner


def run(A, a_dt, desc, buf, K, y_dt, M):
    Y, full = empty_guarded(M * desc.N, y_dt)
    mnb.mnb_matmul_prepacked(to_dev(A, a_dt), desc, buf, Y, K=K, M=M)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(M, desc.N)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("s_dt,with_zp", [("f32", False), ("f16", True), ("bf16", False)])
def test_prepack_bytes_match_the_oracle(bits, bs, s_dt, with_zp):
    N, K = 300, 1000  # a partial last block; rows padded to 16-byte units
    g = wl.rng(seed("pp-bytes", bits, bs, s_dt, with_zp))
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, s_dt, with_zp)
    desc, buf = prepack(packed, scales, s_dt, zp, N, K, bits, bs, identity=0xFEED0000 + bits)
    ref = oracle.prepack(packed, scales, s_dt, zp, N, K, bits, bs, identity=0xFEED0000 + bits)
    assert np.array_equal(buf.cpu().numpy(), ref)
    assert (desc.N, desc.K, desc.bits, desc.block_size, desc.bytes) == (N, K, bits, bs, ref.size)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("a_dt,M,with_zp", [("f32", 1, False), ("f16", 3, True), ("bf16", 5, False),
                                             ("f32", 20, True)])
def test_matmul_prepacked_against_the_oracle(bits, bs, a_dt, M, with_zp):
    N, K = 1000, 1000
    s_dt = "f32" if a_dt == "f32" else a_dt
    g = wl.rng(seed("pp-mm", bits, bs, a_dt, M, with_zp))
    packed, scales, zp = wl.quantized_weight(g, N, K, bits, bs, s_dt, with_zp)
    A = wl.normal(g, (M, K), a_dt)
    desc, buf = prepack(packed, scales, s_dt, zp, N, K, bits, bs)
    y_dt = "f32" if a_dt == "f32" else a_dt
    y = run(A, a_dt, desc, buf, K, y_dt, M)
    ref = oracle.mnb_matmul(A, a_dt, packed, scales, s_dt, zp, N, K, bits, bs, threads=THREADS)
    assert_close(y, ref, y_dt, a_dt)


@pytest.mark.parametrize("bits,bs", [(3, 32), (3, 64), (4, 32)])
def test_vocab_head_decode_prepacked(bits, bs):
    """The Qwen3-1.7B vocabulary head (2048 -> 151936), M = 1, fp32, on sampled rows."""
    K, N = wl.QWEN3_1P7B_LM_HEAD[1:]
    g = wl.rng(seed("pp-head", bits, bs))
    packed, scales, _ = wl.quantized_weight(g, N, K, bits, bs, "f32", False)
    A = wl.normal(g, (1, K), "f32")
    desc, buf = prepack(packed, scales, "f32", None, N, K, bits, bs)
    y = run(A, "f32", desc, buf, K, "f32", 1)
    rows = np.sort(wl.rng(seed("pp-head-rows", bits, bs)).choice(N, 256, replace=False))
    ref = oracle.mnb_matmul(A, "f32", packed[rows], scales[rows], "f32", None, len(rows), K, bits, bs,
                            threads=THREADS)
    assert_close(y[:, rows], ref, "f32")


@pytest.mark.parametrize("bits", [3, 4])
def test_integer_data_is_bit_exact(bits):
    """Integer activations, unit scales, zero points 0: every chunk sum and partial sum
    is an integer below 2^24, so the prepacked path equals the oracle exactly."""
    g = wl.rng(seed("pp-exact", bits))
    N, K, bs, M = 200, 2048, 64, 2
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    scales = np.ones((N, K // bs), np.float32)
    zp = oracle.pack_zero_points(np.zeros((N, K // bs), np.uint8), bits)
    A = g.integers(-3, 4, size=(M, K)).astype(np.float32)
    desc, buf = prepack(packed, scales, "f32", zp, N, K, bits, bs)
    y = run(A, "f32", desc, buf, K, "f32", M)
    assert np.array_equal(y, A.astype(np.float64) @ codes.astype(np.float64).T)


def test_stale_identity_is_refused_on_the_device():
    """A buffer re-prepacked for another weight while the caller still holds the first
    descriptor: the host cannot tell, the kernel checks the device header, records
    MNB_ERR_INVALID_ARG and leaves Y untouched; the current descriptor still works."""
    N, K, bits, bs = 512, 512, 3, 32
    g = wl.rng(seed("pp-stale"))
    p1, s1, _ = wl.quantized_weight(g, N, K, bits, bs, "f32", False)
    p2, s2, _ = wl.quantized_weight(g, N, K, bits, bs, "f32", False)
    A = to_dev(wl.normal(g, (1, K), "f32"))
    n = mnb.mnb_prepack_size(N, K, bits, bs, mnb.F32, False)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    old = mnb.mnb_prepack(to_dev(p1), to_dev(s1), None, N, K, bits, bs, buf, identity=1)
    new = mnb.mnb_prepack(to_dev(p2), to_dev(s2), None, N, K, bits, bs, buf, identity=2)
    torch.cuda.synchronize()
    assert mnb.mnb_get_last_device_error() == 0
    Y = torch.full((N,), 7.0, device="cuda")
    assert mnb.mnb_matmul_prepacked(A, old, buf, Y, K=K, M=1, check=False) == 0  # launched
    torch.cuda.synchronize()
    assert mnb.mnb_status_string(mnb.mnb_get_last_device_error()) == "MNB_ERR_INVALID_ARG"
    assert bool((Y == 7.0).all())
    mnb.mnb_matmul_prepacked(A, new, buf, Y, K=K, M=1)
    torch.cuda.synchronize()
    assert mnb.mnb_get_last_device_error() == 0
    ref = oracle.mnb_matmul(A.cpu().numpy(), "f32", p2, s2, "f32", None, N, K, bits, bs)
    assert_close(to_f64(Y).reshape(1, N), ref, "f32")


def test_descriptor_checks_on_the_host():
    N, K, bits, bs = 64, 256, 4, 32
    g = wl.rng(seed("pp-host"))
    p, s, _ = wl.quantized_weight(g, N, K, bits, bs, "f32", False)
    n = mnb.mnb_prepack_size(N, K, bits, bs, mnb.F32, False)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    desc = mnb.mnb_prepack(to_dev(p), to_dev(s), None, N, K, bits, bs, buf)
    A = torch.zeros((1, K), device="cuda")
    Y = torch.empty(N, device="cuda")
    bad = mnb.PrepackedDesc.from_buffer_copy(desc)
    bad.version = 2
    assert mnb.mnb_status_string(mnb.mnb_matmul_prepacked(A, bad, buf, Y, K=K, M=1, check=False)) == \
        "MNB_ERR_INVALID_ARG"
    assert mnb.mnb_status_string(mnb.mnb_matmul_prepacked(A[:, :128], desc, buf, Y, K=128, M=1, check=False)) == \
        "MNB_ERR_INVALID_ARG"
    small = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    st, _ = mnb.mnb_prepack(to_dev(p), to_dev(s), None, N, K, bits, bs, small, check=False)
    assert mnb.mnb_status_string(st) == "MNB_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert mnb.mnb_get_last_device_error() == 0
