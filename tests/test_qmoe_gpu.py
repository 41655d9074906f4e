"""GPU parity of qmoe_forward (routing, FC1 + SwiGLU, FC2, combine) against the
oracle, through the C ABI.  Outputs are fp16 / bf16:
|y - r| <= 1e-2 + 2e-2 max(|r|, rms(r)) (tests/_util.py)."""
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import assert_half_close, empty_guarded, guards_intact, to_dev, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1
MOE = wl.QWEN3_30B_A3B_MOE


def seed(*key):
    return zlib.crc32(repr(key).encode())


def run_qmoe(d, T, H, I, E, k, b1, b2, bs, act, layout="interleaved", normalize=True):
    code = {"f16": mnb.F16, "bf16": mnb.BF16}[act]
    ws = torch.empty(mnb.qmoe_workspace_size(T, H, I, E, k, code), dtype=torch.uint8, device="cuda")
    Y, full = empty_guarded(T * H, act)
    lay = mnb.FC1_INTERLEAVED if layout == "interleaved" else mnb.FC1_CONCAT
    z = lambda a: None if a is None else to_dev(a)
    mnb.qmoe_forward(to_dev(d["X"], act), to_dev(d["logits"]), k, normalize, to_dev(d["fc1_w"]),
                     to_dev(d["fc1_scales"], act), z(d["fc1_zp"]), b1, to_dev(d["fc2_w"]), to_dev(d["fc2_scales"], act),
                     z(d["fc2_zp"]), b2, I, bs, Y, ws, fc1_layout=lay)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(T, H)


def reference(d, k, b1, b2, I, bs, act, layout="interleaved", normalize=True, tokens=None):
    return oracle.qmoe(d["X"], act, d["logits"], k, normalize, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], b1,
                       d["fc2_w"], d["fc2_scales"], d["fc2_zp"], b2, I, bs, layout, tokens=tokens, threads=THREADS)


def test_int3_decode_layer():
    """One Qwen3-30B-A3B-shaped layer, T=1, (3,3), block 64, fp16, top-8 renormalised."""
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    d = wl.moe_layer(wl.rng(seed("c3")), 1, H, I, E, 3, 3, 64, "f16")
    y = run_qmoe(d, 1, H, I, E, k, 3, 3, 64, "f16")
    assert_half_close(y, reference(d, k, 3, 3, I, 64, "f16"))


@pytest.mark.parametrize("T", [1, 2, 5, 8])
@pytest.mark.parametrize("bits", [(3, 3), (3, 4), (4, 3), (4, 4)])
def test_decode_plan(T, bits):
    b1, b2 = bits
    H, I, E, k, bs = 1024, 512, 64, 8, 64
    act = "bf16" if T % 2 else "f16"
    d = wl.moe_layer(wl.rng(seed("dec", T, bits)), T, H, I, E, b1, b2, bs, act, with_zp=(T == 2))
    y = run_qmoe(d, T, H, I, E, k, b1, b2, bs, act)
    assert_half_close(y, reference(d, k, b1, b2, I, bs, act))


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("normalize", [True, False])
def test_decode_layouts_and_blocks(bs, layout, normalize):
    H, I, E, k, T = 512, 256, 32, 4, 3
    d = wl.moe_layer(wl.rng(seed("lay", bs, layout, normalize)), T, H, I, E, 3, 4, bs, "f16", with_zp=True)
    y = run_qmoe(d, T, H, I, E, k, 3, 4, bs, "f16", layout, normalize)
    assert_half_close(y, reference(d, k, 3, 4, I, bs, "f16", layout, normalize))


@pytest.mark.parametrize("T,E,k,skew", [(9, 64, 8, True), (64, 128, 8, True), (33, 16, 2, False), (40, 8, 8, False),
                                        (12, 1, 1, False), (20, 256, 10, True)])
@pytest.mark.parametrize("bits", [(3, 3), (4, 3)])
def test_tiled_plan(T, E, k, skew, bits):
    b1, b2 = bits
    H, I, bs = 512, 256, 64
    d = wl.moe_layer(wl.rng(seed("tiled", T, E, k, bits)), T, H, I, E, b1, b2, bs, "bf16", with_zp=skew, skew=skew)
    y = run_qmoe(d, T, H, I, E, k, b1, b2, bs, "bf16")
    assert_half_close(y, reference(d, k, b1, b2, I, bs, "bf16"))


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("I,bits", [(128, 4), (96, 4), (96, 3)])
def test_tiled_plan_layouts(layout, I, bits):
    """Both FC1 row layouts; I = 96 leaves the last weight tile of each expert
    half empty (its gate and up rows are read as two 64-row tiles in the
    concatenated layout)."""
    H, E, k, T, bs = 256, 16, 4, 50, 32
    d = wl.moe_layer(wl.rng(seed("tiled-layout", layout, I, bits)), T, H, I, E, bits, bits, bs, "f16", with_zp=True,
                     skew=True)
    y = run_qmoe(d, T, H, I, E, k, bits, bits, bs, "f16", layout)
    assert_half_close(y, reference(d, k, bits, bits, I, bs, "f16", layout))


@pytest.mark.parametrize("T", [128, 512])
def test_prefill_shapes_sampled_tokens(T):
    """Qwen3-30B-A3B-shaped layer, skewed routing; every output of a sample of tokens."""
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    d = wl.moe_layer(wl.rng(seed("prefill", T)), T, H, I, E, 3, 3, 64, "f16", skew=True)
    y = run_qmoe(d, T, H, I, E, k, 3, 3, 64, "f16")
    toks = sorted(set([0, 1, T - 1, 10, 20] + list(wl.rng(T).integers(0, T, 11))))
    assert_half_close(y[toks], reference(d, k, 3, 3, I, 64, "f16", tokens=toks))


@pytest.mark.parametrize("T,bits,bs,act,zp", [(2048, (3, 3), 64, "f16", False), (4096, (4, 4), 32, "bf16", True),
                                              (4096, (3, 4), 128, "f16", True), (2048, (4, 3), 64, "bf16", False)])
def test_prefill_sweep_full_size_sampled_tokens(T, bits, bs, act, zp):
    """Full-size prefill sweep points (Qwen3-30B-A3B layer, 10% of tokens skewed onto
    experts 0-7): every output of a sample of tokens against the oracle."""
    b1, b2 = bits
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    d = wl.moe_layer(wl.rng(seed("sweep", T, bits, bs, act, zp)), T, H, I, E, b1, b2, bs, act, with_zp=zp,
                     skew=True)
    y = run_qmoe(d, T, H, I, E, k, b1, b2, bs, act)
    toks = sorted(set([0, 10, T - 1] + list(wl.rng(T + 1).integers(0, T, 7))))
    assert_half_close(y[toks], reference(d, k, b1, b2, I, bs, act, tokens=toks))
