"""GPU parity of mnb_gate_up_swiglu (the dense FFN's gate and up projections
fused with SwiGLU) against the oracle, through the C ABI: the CUDA-core path
(M < 16, or fp32 activations / outputs) and the tensor-core path (M >= 16,
16-bit activations and output), both gate/up layouts."""
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import (assert_close, assert_swiglu_bf16_tc_close, assert_swiglu_f32_close, empty_guarded,
                         guards_intact, to_dev, to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1
LAYOUT = {"interleaved": mnb.FC1_INTERLEAVED, "concat": mnb.FC1_CONCAT}


def seed(*key):
    return zlib.crc32(repr(key).encode())


def make(g, M, K, I, bits, bs, a_dt, s_dt, with_zp):
    packed, scales, zp = wl.quantized_weight(g, 2 * I, K, bits, bs, s_dt, with_zp)
    A = wl.normal(g, (M, K), a_dt)
    return A, packed, scales, zp


def gate_and_up(A, a_dt, packed, scales, s_dt, zp, I, K, bits, bs, layout):
    """The oracle's gate and up products [M, I] each, from the plain matmul over
    the 2I rows in their layout."""
    both = oracle.mnb_matmul(A, a_dt, packed, scales, s_dt, zp, 2 * I, K, bits, bs, threads=THREADS)
    if layout == "interleaved":
        return both[:, 0::2], both[:, 1::2]
    return both[:, :I], both[:, I:]


def check(y, y_dt, a_dt, A, packed, scales, s_dt, zp, I, K, bits, bs, layout, tensor_cores=False, label=""):
    if y_dt == "f32" or (tensor_cores and y_dt == "bf16" and a_dt == "bf16"):
        # fp32 outputs and bf16 tensor-core outputs: the rule of a plain product
        # on the gate and up products, carried through SwiGLU by its
        # first-order sensitivity (a large |u| magnifies the gate's error)
        g, u = gate_and_up(A, a_dt, packed, scales, s_dt, zp, I, K, bits, bs, layout)
        if y_dt == "f32":
            assert_swiglu_f32_close(y, g, u, label=label)
        else:
            assert_swiglu_bf16_tc_close(y, g, u, label=label)
    else:
        ref = oracle.gate_up_swiglu(A, a_dt, packed, scales, s_dt, zp, I, K, bits, bs, layout, threads=THREADS)
        assert_close(y, ref, y_dt, a_dt, tensor_cores=tensor_cores, label=label)


def run(A, a_dt, packed, scales, s_dt, zp, I, K, bits, bs, layout, y_dt, M):
    Y, full = empty_guarded(M * I, y_dt)
    mnb.mnb_gate_up_swiglu(to_dev(A, a_dt), to_dev(packed), to_dev(scales, s_dt),
                           None if zp is None else to_dev(zp), I, bits, bs, Y, layout=LAYOUT[layout], K=K, M=M)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(M, I)


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
def test_qwen3_dense_mlp_decode(layout):
    """One token through the Qwen3-1.7B MLP's gate/up (K 2048, I 6144), INT4, block 32."""
    K, I = 2048, 6144
    g = wl.rng(seed("gate-up-decode", layout))
    A, packed, scales, zp = make(g, 1, K, I, 4, 32, "f32", "f32", False)
    y = run(A, "f32", packed, scales, "f32", None, I, K, 4, 32, layout, "f32", 1)
    check(y, "f32", "f32", A, packed, scales, "f32", None, I, K, 4, 32, layout, label=f"gate/up decode {layout}")


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("a_dt,M", [("f16", 1), ("bf16", 3), ("f32", 20)])
def test_formats_cuda_cores(bits, bs, layout, a_dt, M):
    """Every width and block size with zero points, a partial last K block and an I
    that ends inside a block of pairs; fp32 activations at M = 20 stay on CUDA cores."""
    K, I = 1000, 333
    g = wl.rng(seed("gate-up-fmt", bits, bs, layout, a_dt, M))
    A, packed, scales, zp = make(g, M, K, I, bits, bs, a_dt, "f32", True)
    y_dt = "f32" if a_dt == "f32" else a_dt
    y = run(A, a_dt, packed, scales, "f32", zp, I, K, bits, bs, layout, y_dt, M)
    check(y, y_dt, a_dt, A, packed, scales, "f32", zp, I, K, bits, bs, layout, label=f"gate/up {a_dt} M={M}")


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("a_dt", ["f16", "bf16"])
@pytest.mark.parametrize("M,with_zp", [(16, False), (300, True)])
def test_tensor_cores(bits, layout, a_dt, M, with_zp):
    """M >= 16 with 16-bit activations: the tensor-core FC1 tiles over the dense matrix
    (a ragged last 256-row tile at M = 300, I = 1000 ends inside a 64-pair tile),
    16-bit scales."""
    K, I, bs = 1024, 1000, 64
    g = wl.rng(seed("gate-up-tc", bits, layout, a_dt, M, with_zp))
    A, packed, scales, zp = make(g, M, K, I, bits, bs, a_dt, a_dt, with_zp)
    y = run(A, a_dt, packed, scales, a_dt, zp, I, K, bits, bs, layout, a_dt, M)
    check(y, a_dt, a_dt, A, packed, scales, a_dt, zp, I, K, bits, bs, layout, tensor_cores=True,
          label=f"gate/up tc M={M} {a_dt} {layout}")


def test_layouts_agree_bit_for_bit():
    """The same weights stored interleaved and concatenated give the same bits (each
    output's gate and up dot products run over the same values in the same order)."""
    K, I, bits, bs = 2048, 512, 4, 32
    g = wl.rng(seed("gate-up-layouts"))
    A, packed, scales, _ = make(g, 2, K, I, bits, bs, "bf16", "f32", False)
    row_b, nb = packed.shape[1], scales.shape[1]
    cat_p = np.concatenate([packed[0::2], packed[1::2]]).reshape(2 * I, row_b)
    cat_s = np.concatenate([scales[0::2], scales[1::2]]).reshape(2 * I, nb)
    y_i = run(A, "bf16", packed, scales, "f32", None, I, K, bits, bs, "interleaved", "f32", 2)
    y_c = run(A, "bf16", cat_p, cat_s, "f32", None, I, K, bits, bs, "concat", "f32", 2)
    assert np.array_equal(y_i, y_c)


def test_concat_needs_whole_16_byte_rows_on_cuda_cores():
    """K 96 at block 32 with 16-bit scales: 6-byte scale rows cannot be staged by the
    separate gate/up bulk copies; the interleaved layout of the same weights runs."""
    K, I, bits, bs = 96, 64, 3, 32
    g = wl.rng(seed("gate-up-unsupported"))
    A, packed, scales, _ = make(g, 1, K, I, bits, bs, "f16", "f16", False)
    Y = torch.empty(I, dtype=torch.float16, device="cuda")
    st = mnb.mnb_gate_up_swiglu(to_dev(A, "f16"), to_dev(packed), to_dev(scales, "f16"), None, I, bits, bs, Y,
                                layout=mnb.FC1_CONCAT, K=K, M=1, check=False)
    assert mnb.mnb_status_string(st) == "MNB_ERR_UNSUPPORTED"
    y = run(A, "f16", packed, scales, "f16", None, I, K, bits, bs, "interleaved", "f16", 1)
    ref = oracle.gate_up_swiglu(A, "f16", packed, scales, "f16", None, I, K, bits, bs, "interleaved")
    assert_close(y, ref, "f16")
