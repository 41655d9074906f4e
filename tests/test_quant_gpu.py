"""GPU parity of mnb_quantize_int3 (symmetric grouped INT3 round-to-nearest, the
producer policy quoted in "INT3 QMoE CUDA correctness baseline and Qwen
experimental results") against the oracle: packed bytes and scale bit patterns
are compared exactly, since every code is an integer decided in binary32 on
both sides."""
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import assert_f32_close, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

SD = {"f32": mnb.F32, "f16": mnb.F16, "bf16": mnb.BF16}


def seed(*key):
    return zlib.crc32(repr(key).encode())


def weights(g, N, K, bs):
    """Normal weights with per-row magnitudes over fifteen decades (so that
    binary16 scales run from underflow through subnormals to overflow), plus an
    all-zero block, a block of exact ties (max|w| = 3.5 * 2^-3, every quotient a
    half-integer) and a block holding +-max|w|."""
    mag = (10.0 ** g.uniform(-7, 3, size=N)).astype(np.float32)
    w = (g.standard_normal((N, K)).astype(np.float32) * mag[:, None]).astype(np.float32)
    w[0, :bs] = 0.0
    if N > 1:
        ties = (g.integers(-4, 3, size=bs) + 0.5).astype(np.float32) * np.float32(0.125)
        ties[0] = np.float32(3.5 * 0.125)
        w[1, :bs] = ties
    if N > 2:
        w[2, bs - 1] = np.abs(w[2, :bs]).max() * 2
        w[2, 0] = -w[2, bs - 1]
    return w


def run(w32, w_dtype, bs, s_dtype):
    W = to_dev(wl.cast(w32, w_dtype), w_dtype)
    B, S = mnb.mnb_quantize_int3(W, bs, SD[s_dtype])
    status = mnb.mnb_get_last_device_error()
    B = B.cpu().numpy().reshape(w32.shape[0], -1)
    S = S.cpu().view(torch.int32 if s_dtype == "f32" else torch.int16).numpy()
    return B, S, status


def ref(w32, w_dtype, bs, s_dtype):
    packed, scales, bad = oracle.quantize_int3(wl.cast(w32, w_dtype), w_dtype, bs, s_dtype)
    return packed, scales.view(np.int32 if s_dtype == "f32" else np.int16), bad


@pytest.mark.parametrize("N,K,bs", [(5, 256, 32), (33, 2048, 64), (7, 768, 128), (130, 640, 32), (3, 96, 32)])
@pytest.mark.parametrize("w_dtype,s_dtype", [("f32", "f16"), ("f16", "f16"), ("bf16", "bf16"), ("f32", "f32"),
                                             ("f32", "bf16")])
def test_bit_exact_against_oracle(N, K, bs, w_dtype, s_dtype):
    g = wl.rng(seed("quant", N, K, bs, w_dtype, s_dtype))
    w = weights(g, N, K, bs)
    B, S, status = run(w, w_dtype, bs, s_dtype)
    P, R, bad = ref(w, w_dtype, bs, s_dtype)
    assert np.array_equal(B, P)
    assert np.array_equal(S, R)
    assert status == (7 if bad.any() else 0)


def test_rejected_blocks_leave_the_others_intact():
    g = wl.rng(seed("quant-bad"))
    N, K, bs = 6, 256, 64
    w = g.standard_normal((N, K)).astype(np.float32)
    w[1, 70] = np.nan
    w[3, 200] = -np.inf
    w[4, :64] = 1e-9  # the binary16 scale rounds to zero
    w[5, :64] = 3.5e-6  # a subnormal binary16 scale, kept
    B, S, status = run(w, "f32", bs, "f16")
    P, R, bad = ref(w, "f32", bs, "f16")
    assert bad.sum() == 3 and bad[1, 1] and bad[3, 3] and bad[4, 0] and not bad[5, 0]
    assert status == 7  # MNB_ERR_CONTENT
    assert np.array_equal(B, P) and np.array_equal(S, R)
    assert mnb.mnb_get_last_device_error() == 0  # read and cleared


def test_full_size_expert_stack_sampled_rows():
    """FC1 weights of 16 Qwen3-30B-A3B experts (16 x 1536 rows, K = 2048, bs 64,
    fp16 weights and scales) in one call; sampled rows against the oracle, and
    the codes feed mnb_matmul unchanged."""
    g = wl.rng(seed("quant-full"))
    E, R, K, bs = 16, 1536, 2048, 64
    N = E * R
    w = (g.standard_normal((N, K)).astype(np.float32) * np.float32(0.02))
    W = to_dev(wl.cast(w, "f16"), "f16")
    B, S = mnb.mnb_quantize_int3(W, bs, mnb.F16)
    assert mnb.mnb_get_last_device_error() == 0
    rows = np.unique(np.concatenate([[0, N - 1, R - 1, R], g.integers(0, N, size=40)]))
    P, Rs, bad = oracle.quantize_int3(wl.cast(w[rows], "f16"), "f16", bs, "f16")
    assert not bad.any()
    assert np.array_equal(B.reshape(N, -1)[torch.from_numpy(rows).cuda()].cpu().numpy(), P)
    assert np.array_equal(S[torch.from_numpy(rows).cuda()].cpu().view(torch.int16).numpy(), Rs.view(np.int16))
    # the produced tensors are a valid INT3 projection for the matmul path (seeded
    # activations; the fp32 rule against the oracle's product of the sampled rows)
    a = wl.normal(g, (1, K), "f32")
    A = to_dev(a)
    Y = torch.empty((1, N), device="cuda")
    mnb.mnb_matmul(A, B, S.float(), None, N, 3, bs, Y)
    assert mnb.mnb_get_last_device_error() == 0
    y_ref = oracle.mnb_matmul(a, "f32", P, Rs, "f16", None, rows.size, K, 3, bs)
    assert_f32_close(Y[0, torch.from_numpy(rows).cuda()].cpu().double().numpy()[None, :], y_ref)


@pytest.mark.parametrize("w_dtype,s_dtype", [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16"), ("f32", "f16")])
def test_exact_ties_at_scale(w_dtype, s_dtype):
    """Weights on a coarse grid (small integers times 2^-7) make w / scale an
    exact half-integer for many codes, so the ties-to-even decision is taken
    ~200 000 times per case (a quarter of the rows are plain normal weights);
    4M weights compared with the oracle byte for byte."""
    g = wl.rng(seed("quant-ties", w_dtype, s_dtype))
    N, K, bs = 2048, 2048, 64
    w = (g.integers(-56, 57, size=(N, K)).astype(np.float32) * np.float32(2.0 ** -7))
    w[: N // 2] *= np.float32(1.0) + g.integers(0, 4, size=(N // 2, 1)).astype(np.float32) / np.float32(8)
    w[N // 2: 3 * N // 4] = g.standard_normal((N // 4, K)).astype(np.float32) * np.float32(0.02)
    B, S, status = run(w, w_dtype, bs, s_dtype)
    P, R, bad = ref(w, w_dtype, bs, s_dtype)
    assert not bad.any() and status == 0
    assert np.array_equal(S, R)
    assert np.array_equal(B, P)
