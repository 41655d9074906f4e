"""qmoe_forward_static: the QMoE layer for callers that cannot allocate device
memory (plugins that only receive input/output pointers, runtimes that own every
allocation, code that must not call cudaMalloc on its path).  It runs the same
kernels as qmoe_forward with the library's fixed 8 MiB scratch array instead of a
caller workspace.  This file is named to be collected last."""
import zlib

import numpy as np
import pytest

import workloads as wl
from tests._util import to_dev, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

MOE = wl.QWEN3_30B_A3B_MOE


def layer(seed, T, b1=3, b2=3, bs=64, act="f16"):
    H, I, E = MOE["H"], MOE["I"], MOE["E"]
    d = wl.moe_layer(wl.rng(seed), T, H, I, E, b1, b2, bs, act, with_zp=(T > 1), skew=True)
    dev = {key: (None if v is None else to_dev(v, act if "scales" in key or key == "X" else None))
           for key, v in d.items()}
    return dev, (H, I, E, b1, b2, bs, act)


def with_workspace(dev, shape, T, k):
    H, I, E, b1, b2, bs, act = shape
    code = mnb.F16 if act == "f16" else mnb.BF16
    ws = torch.empty(mnb.qmoe_workspace_size(T, H, I, E, k, code), dtype=torch.uint8, device="cuda")
    Y = torch.empty((T, H), dtype=torch.float16 if act == "f16" else torch.bfloat16, device="cuda")
    mnb.qmoe_forward(dev["X"], dev["logits"], k, True, dev["fc1_w"], dev["fc1_scales"], dev["fc1_zp"], b1,
                     dev["fc2_w"], dev["fc2_scales"], dev["fc2_zp"], b2, I, bs, Y, ws)
    return Y


def static(dev, shape, T, k):
    H, I, E, b1, b2, bs, act = shape
    Y = torch.empty((T, H), dtype=torch.float16 if act == "f16" else torch.bfloat16, device="cuda")
    mnb.qmoe_forward_static(dev["X"], dev["logits"], k, True, dev["fc1_w"], dev["fc1_scales"], dev["fc1_zp"], b1,
                            dev["fc2_w"], dev["fc2_scales"], dev["fc2_zp"], b2, I, bs, Y)
    return Y


@pytest.mark.parametrize("T,bits,act", [(1, (3, 3), "f16"), (5, (4, 3), "bf16"), (40, (3, 4), "f16")])
def test_static_scratch_matches_workspace_on_two_calls_in_a_row(T, bits, act):
    """Same kernels, same inputs: the static-scratch call must equal the
    workspace call bit for bit.  Before the pair of calls a larger layer (90
    tokens) fills the scratch with its own tables and activations, so stale
    contents from an earlier call would show."""
    k = MOE["k"]
    first, shape = layer(zlib.crc32(repr(("static-a", T, bits, act)).encode()), T, *bits, act=act)
    second, _ = layer(zlib.crc32(repr(("static-b", T, bits, act)).encode()), T, *bits, act=act)
    filler, fshape = layer(zlib.crc32(repr(("static-fill", T, bits, act)).encode()), 90, *bits, act=act)
    static(filler, fshape, 90, k)
    ys = [static(first, shape, T, k), static(second, shape, T, k)]   # two calls in a row, same scratch
    torch.cuda.synchronize()
    assert mnb.mnb_get_last_device_error() == 0
    refs = [with_workspace(first, shape, T, k), with_workspace(second, shape, T, k)]
    torch.cuda.synchronize()
    for y, r in zip(ys, refs):
        assert torch.equal(y, r)
    assert not np.array_equal(to_f64(ys[0]), to_f64(ys[1]))   # the second call did not reuse stale results


def test_static_scratch_rejects_problems_beyond_its_size():
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    X = torch.zeros((93, H), dtype=torch.float16, device="cuda")   # 93 tokens need more than 8 MiB of scratch
    st = mnb.qmoe_forward_static(X, torch.zeros((93, E), device="cuda"), k, True, 16, 16, None, 3, 16, 16, None, 3, I,
                                 64, torch.empty_like(X), check=False)
    assert st == 4  # MNB_ERR_WORKSPACE
