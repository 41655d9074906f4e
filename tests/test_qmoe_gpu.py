"""GPU parity of qmoe_forward (routing, FC1 + SwiGLU, FC2, combine) against the
oracle, through the C ABI.  Outputs are fp16 / bf16: the elementwise rule
|y - r| <= 1e-2 + 2e-2 |r|, except bf16 layers with T > 8 (which may run on the
tensor-core plan), which take the bf16 tensor-core rule and print their
elementwise misses (tests/_util.py); the grouped CUDA-core plan's own tests
hold it to the elementwise rule.  Sampled prefill checks cover at least 64
tokens.  Plans: one token -> the single-pass layer; two tokens (and up to 8
where the grouped plan does not apply) -> the two-kernel decode; from 3 tokens
with up to 1.5 routed rows per expert on average, or X rows off a 16-byte
boundary -> the grouped CUDA-core plan (m-tiles of <= 4 rows, one GEMV ring per
expert block); more -> the tensor-core plan; the tiled CUDA-core plan takes
what the grouped plan cannot (concatenated gate/up rows whose bytes or scales
are not whole 16-byte units, with X rows off a 16-byte boundary)."""
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
MOE = wl.QWEN3_30B_A3B_MOE


def seed(*key):
    return zlib.crc32(repr(key).encode())


def run_qmoe(d, T, H, I, E, k, b1, b2, bs, act, layout="interleaved", normalize=True):
    code = {"f16": mnb.F16, "bf16": mnb.BF16}[act]
    ws, ws_full = guarded_workspace(mnb.qmoe_workspace_size(T, H, I, E, k, code))
    Y, full = empty_guarded(T * H, act)
    lay = mnb.FC1_INTERLEAVED if layout == "interleaved" else mnb.FC1_CONCAT
    z = lambda a: None if a is None else to_dev(a)
    mnb.qmoe_forward(to_dev(d["X"], act), to_dev(d["logits"]), k, normalize, to_dev(d["fc1_w"]),
                     to_dev(d["fc1_scales"], act), z(d["fc1_zp"]), b1, to_dev(d["fc2_w"]), to_dev(d["fc2_scales"], act),
                     z(d["fc2_zp"]), b2, I, bs, Y, ws, fc1_layout=lay)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert guards_intact(ws_full, 256), "write outside the workspace"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(T, H)


def check(y, ref, act, T, label=""):
    """The rule of the plan that ran: T > 8 is the tensor-core plan."""
    assert_close(y, ref, act, act, tensor_cores=T > 8, label=label)


def sample_tokens(T, key, n=64):
    """Every token up to n, else the first, last and tenth plus random distinct ones, n in all."""
    if T <= n:
        return list(range(T))
    g = wl.rng(seed(*key))
    toks = {0, 10, T - 1}
    while len(toks) < n:
        toks.add(int(g.integers(0, T)))
    return sorted(toks)


def reference(d, k, b1, b2, I, bs, act, layout="interleaved", normalize=True, tokens=None):
    return oracle.qmoe(d["X"], act, d["logits"], k, normalize, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], b1,
                       d["fc2_w"], d["fc2_scales"], d["fc2_zp"], b2, I, bs, layout, tokens=tokens, threads=THREADS)


def test_int3_decode_layer():
    """One Qwen3-30B-A3B-shaped layer, T=1, (3,3), block 64, fp16, top-8 renormalised."""
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    d = wl.moe_layer(wl.rng(seed("c3")), 1, H, I, E, 3, 3, 64, "f16")
    y = run_qmoe(d, 1, H, I, E, k, 3, 3, 64, "f16")
    check(y, reference(d, k, 3, 3, I, 64, "f16"), "f16", 1)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
@pytest.mark.parametrize("bits", [(3, 3), (3, 4), (4, 3), (4, 4)])
def test_decode_plan(T, bits):
    """T = 1: the single-pass layer; T = 2: the two-kernel decode; T = 5, 8: the
    grouped CUDA-core plan (under one routed row per expert)."""
    b1, b2 = bits
    H, I, E, k, bs = 1024, 512, 64, 8, 64
    act = "bf16" if T % 2 else "f16"
    d = wl.moe_layer(wl.rng(seed("dec", T, bits)), T, H, I, E, b1, b2, bs, act, with_zp=(T == 2))
    y = run_qmoe(d, T, H, I, E, k, b1, b2, bs, act)
    check(y, reference(d, k, b1, b2, I, bs, act), act, T)


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("normalize", [True, False])
def test_decode_layouts_and_blocks(bs, layout, normalize):
    """The two-kernel decode plan (T = 2): both FC1 layouts, every block size."""
    H, I, E, k, T = 512, 256, 32, 4, 2
    d = wl.moe_layer(wl.rng(seed("lay", bs, layout, normalize)), T, H, I, E, 3, 4, bs, "f16", with_zp=True)
    y = run_qmoe(d, T, H, I, E, k, 3, 4, bs, "f16", layout, normalize)
    check(y, reference(d, k, 3, 4, I, bs, "f16", layout, normalize), "f16", T)


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("bs,bits,E,k", [(32, (3, 4), 64, 8), (64, (4, 3), 300, 6), (128, (4, 4), 16, 2),
                                        (64, (3, 3), 128, 8)])
def test_one_token_single_pass(layout, bs, bits, E, k):
    """T = 1 runs the single-pass layer kernel (every CTA's FC1 and FC2 rows copied
    before the dependency wait, a grid barrier between FC1 and FC2): both FC1 layouts,
    explicit zero points, routers wider than one CTA's ranking (E = 300)."""
    b1, b2 = bits
    H, I = 1024, 256 if bs != 128 else 512
    d = wl.moe_layer(wl.rng(seed("one", layout, bs, bits, E, k)), 1, H, I, E, b1, b2, bs, "bf16", with_zp=True)
    y = run_qmoe(d, 1, H, I, E, k, b1, b2, bs, "bf16", layout)
    check(y, reference(d, k, b1, b2, I, bs, "bf16", layout), "bf16", 1)


@pytest.mark.parametrize("T,E,k,skew,cuda_cores", [(9, 64, 8, True, True), (64, 128, 8, True, False),
                                                   (33, 16, 2, False, False), (40, 8, 8, False, False),
                                                   (12, 1, 1, False, False), (20, 256, 10, True, True)])
@pytest.mark.parametrize("bits", [(3, 3), (4, 3)])
def test_small_prefill_layers(T, E, k, skew, cuda_cores, bits):
    """Small layers past the decode range: the grouped CUDA-core plan where the
    routed rows average at most 1.5 per expert (T=9 of 64 experts, T=20 of 256;
    held to the elementwise rule), the tensor-core plan elsewhere (one expert,
    two, eight, sixteen)."""
    b1, b2 = bits
    H, I, bs = 512, 256, 64
    d = wl.moe_layer(wl.rng(seed("tiled", T, E, k, bits)), T, H, I, E, b1, b2, bs, "bf16", with_zp=skew, skew=skew)
    y = run_qmoe(d, T, H, I, E, k, b1, b2, bs, "bf16")
    check(y, reference(d, k, b1, b2, I, bs, "bf16"), "bf16", 1 if cuda_cores else T, f"T={T} E={E} k={k} bits={bits}")


@pytest.mark.parametrize("layout", ["interleaved", "concat"])
@pytest.mark.parametrize("I,bits", [(128, 4), (96, 4), (96, 3)])
def test_tensor_core_plan_layouts(layout, I, bits):
    """The tensor-core plan (12.5 routed rows per expert) in both FC1 row layouts; I = 96 leaves the last weight tile of each expert
    half empty (its gate and up rows are read as two 64-row tiles in the
    concatenated layout)."""
    H, E, k, T, bs = 256, 16, 4, 50, 32
    d = wl.moe_layer(wl.rng(seed("tiled-layout", layout, I, bits)), T, H, I, E, bits, bits, bs, "f16", with_zp=True,
                     skew=True)
    y = run_qmoe(d, T, H, I, E, k, bits, bits, bs, "f16", layout)
    check(y, reference(d, k, bits, bits, I, bs, "f16", layout), "f16", T)


@pytest.mark.parametrize("T", [128, 512])
def test_prefill_shapes_sampled_tokens(T):
    """Qwen3-30B-A3B-shaped layer, skewed routing; every output of a sample of tokens."""
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    d = wl.moe_layer(wl.rng(seed("prefill", T)), T, H, I, E, 3, 3, 64, "f16", skew=True)
    y = run_qmoe(d, T, H, I, E, k, 3, 3, 64, "f16")
    toks = sample_tokens(T, ("prefill", T))
    check(y[toks], reference(d, k, 3, 3, I, 64, "f16", tokens=toks), "f16", T)


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
    toks = sample_tokens(T, ("sweep", T, bits, bs, act, zp))
    check(y[toks], reference(d, k, b1, b2, I, bs, act, tokens=toks), act, T, f"T={T} bits={bits} bs={bs} zp={zp}")


# ------------------------------------------------ producers right ahead of a layer

def test_router_logits_written_by_the_kernel_right_ahead():
    """The router projection (mnb_matmul, M=1, fp32 logits) runs immediately before
    the decode layer on the same stream; the GEMV releases its dependents before it
    writes the logits, so the layer must not read them before its dependency wait."""
    H, I, E, k = MOE["H"], MOE["I"], MOE["E"], MOE["k"]
    g = wl.rng(seed("chain-router"))
    d = wl.moe_layer(g, 1, H, I, E, 3, 3, 64, "f16")
    rw, rs, _ = wl.quantized_weight(g, E, H, 4, 32)          # router weights: INT4 [E, H]
    Xf = torch.from_numpy(d["X"].view(np.int16)).view(torch.float16).float().numpy()
    ws = torch.empty(mnb.qmoe_workspace_size(1, H, I, E, k, mnb.F16), dtype=torch.uint8, device="cuda")
    X_d, X32 = to_dev(d["X"], "f16"), to_dev(Xf)
    W1, S1, W2, S2 = to_dev(d["fc1_w"]), to_dev(d["fc1_scales"], "f16"), to_dev(d["fc2_w"]), to_dev(d["fc2_scales"], "f16")
    RW, RS = to_dev(rw), to_dev(rs)
    logits = torch.full((1, E), float("nan"), device="cuda")   # stale contents would route on NaN
    Y = torch.empty((1, H), dtype=torch.float16, device="cuda")
    for _ in range(3):
        logits.fill_(float("nan"))
        mnb.mnb_matmul(X32, RW, RS, None, E, 4, 32, logits, K=H, M=1)
        mnb.qmoe_forward(X_d, logits, k, True, W1, S1, None, 3, W2, S2, None, 3, I, 64, Y, ws)
        torch.cuda.synchronize()
        assert mnb.mnb_get_last_device_error() == 0
        lg = logits.cpu().numpy()
        d2 = dict(d, logits=lg)
        check(to_f64(Y), reference(d2, k, 3, 3, I, 64, "f16"), "f16", 1)


def test_expert_weights_written_by_the_quantizer_right_ahead():
    """mnb_quantize_int3 writes FC1's packed weights and scales immediately before the
    decode layer that consumes them, on the same stream."""
    H, I, E, k, bs = 1024, 256, 16, 4, 64
    g = wl.rng(seed("chain-quant"))
    d = wl.moe_layer(g, 1, H, I, E, 3, 3, bs, "f16")
    Wd = torch.from_numpy((g.standard_normal((E * 2 * I, H)) * 0.02).astype(np.float16)).cuda()
    W1 = torch.full((E * 2 * I, H // bs, 3 * bs // 8), 0xFF, dtype=torch.uint8, device="cuda")
    S1 = torch.full((E * 2 * I, H // bs), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(mnb.qmoe_workspace_size(1, H, I, E, k, mnb.F16), dtype=torch.uint8, device="cuda")
    Y = torch.empty((1, H), dtype=torch.float16, device="cuda")
    mnb.mnb_quantize_int3(Wd, bs, mnb.F16, W1, S1)
    mnb.qmoe_forward(to_dev(d["X"], "f16"), to_dev(d["logits"]), k, True, W1, S1, None, 3, to_dev(d["fc2_w"]),
                     to_dev(d["fc2_scales"], "f16"), None, 3, I, bs, Y, ws)
    torch.cuda.synchronize()
    assert mnb.mnb_get_last_device_error() == 0
    d2 = dict(d, fc1_w=W1.cpu().numpy().reshape(E, 2 * I, -1),
              fc1_scales=S1.cpu().view(torch.int16).numpy().view(np.uint16).reshape(E, 2 * I, -1))
    check(to_f64(Y), reference(d2, k, 3, 3, I, bs, "f16"), "f16", 1)


# ----------------------------------------------------------- optional inputs

def run_qmoe_ex(d, T, H, I, E, k, b1, b2, bs, act, layout, b1v, b2v, agg, ldt, x_offset=0):
    """qmoe_forward_ex; x_offset = 1 places X one element past a 16-byte boundary
    (its rows then cannot be read with 16-byte loads: the tiled CUDA-core plan)."""
    code = {"f16": mnb.F16, "bf16": mnb.BF16}[act]
    ws, ws_full = guarded_workspace(mnb.qmoe_workspace_size(T, H, I, E, k, code))
    Y, full = empty_guarded(T * H, act)
    Xbuf = torch.zeros(T * H + 8, dtype=torch.float16 if act == "f16" else torch.bfloat16, device="cuda")
    Xbuf[x_offset:x_offset + T * H] = to_dev(d["X"], act).reshape(-1)
    X = Xbuf[x_offset:x_offset + T * H]
    z = lambda a: None if a is None else to_dev(a)
    lay = mnb.FC1_INTERLEAVED if layout == "interleaved" else mnb.FC1_CONCAT
    mnb.qmoe_forward_ex(X, to_dev(d["logits"], ldt if ldt != "f32" else None), k, True, to_dev(d["fc1_w"]),
                        to_dev(d["fc1_scales"], act), z(d["fc1_zp"]), b1, to_dev(d["fc2_w"]), to_dev(d["fc2_scales"], act),
                        z(d["fc2_zp"]), b2, I, bs, Y, ws, fc1_bias=None if b1v is None else to_dev(b1v, act),
                        fc2_bias=None if b2v is None else to_dev(b2v, act), agg_weights=None if agg is None else to_dev(agg),
                        fc1_layout=lay, T=T, H=H, E=E, act_dtype=code)
    torch.cuda.synchronize()
    assert guards_intact(full), "write outside Y"
    assert guards_intact(ws_full, 256), "write outside the workspace"
    assert mnb.mnb_get_last_device_error() == 0
    return to_f64(Y).reshape(T, H)


@pytest.mark.parametrize("T,x_offset", [(1, 0), (2, 0), (12, 0), (40, 0), (20, 1)])
@pytest.mark.parametrize("opts", ["biases", "agg", "half_logits", "all"])
@pytest.mark.parametrize("layout", ["interleaved", "concat"])
def test_optional_inputs_every_plan(T, x_offset, opts, layout):
    """FC1/FC2 biases, aggregation weights and 16-bit router logits on every plan: the
    single-pass layer (T = 1), the two-kernel decode (T = 2), the grouped CUDA-core
    plan (T = 12: 1.5 routed rows per expert; T = 20 with X rows off a 16-byte
    boundary) and the tensor-core plan (T = 40: 5 rows per expert)."""
    H, I, E, k, bs, b1, b2 = 512, 256, 32, 4, 64, 3, 4
    act = "bf16" if T % 2 else "f16"
    g = wl.rng(seed("opts", T, x_offset, opts, layout))
    d = wl.moe_layer(g, T, H, I, E, b1, b2, bs, act, with_zp=True, skew=True)
    want_b = opts in ("biases", "all")
    b1v = wl.normal(g, (E, 2 * I), act) if want_b else None
    b2v = wl.normal(g, (E, H), act) if want_b else None
    agg = wl.uniform(g, (T, E), 0.0, 1.0) if opts in ("agg", "all") else None
    ldt = "bf16" if opts in ("half_logits", "all") else "f32"
    if ldt != "f32":
        d = dict(d, logits=wl.cast(d["logits"], ldt))
    y = run_qmoe_ex(d, T, H, I, E, k, b1, b2, bs, act, layout, b1v, b2v, agg, ldt, x_offset)
    ref = oracle.qmoe_ex(d["X"], act, d["logits"], ldt, k, True, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], b1v, b1,
                         d["fc2_w"], d["fc2_scales"], d["fc2_zp"], b2v, b2, I, bs, layout, agg=agg, threads=THREADS)
    check(y, ref, act, T if x_offset == 0 else 1, f"opts={opts} T={T} layout={layout}")


# ---------------------------------------------------- grouped CUDA-core plan

@pytest.mark.parametrize("T,E,k,layout,bits,bs,act,zp,x_offset", [
    (16, 128, 8, "interleaved", (3, 3), 64, "bf16", True, 0),   # 1 routed row per expert on average
    (12, 32, 4, "concat", (4, 3), 32, "f16", False, 0),          # 1.5: the largest mean it takes
    (24, 32, 2, "interleaved", (4, 4), 128, "bf16", True, 0),
    (9, 1, 1, "concat", (3, 4), 64, "f16", True, 1),             # one expert: 3 m-tiles, the last of 1 row
    (300, 8, 2, "interleaved", (3, 4), 64, "f16", True, 1),      # X off 16 bytes: any mean (75 rows per expert)
    (50, 64, 6, "concat", (3, 3), 64, "bf16", True, 1),
])
def test_grouped_plan(T, E, k, layout, bits, bs, act, zp, x_offset):
    """The grouped CUDA-core plan (exact dp4a chunk sums, fp32 accumulation) against
    the oracle under the elementwise 16-bit rule, both FC1 layouts, zero points,
    skewed routing (ragged m-tiles) and biases."""
    b1, b2 = bits
    H, I = 1024, 512
    g = wl.rng(seed("grouped", T, E, k, layout, bits, bs, act, zp, x_offset))
    d = wl.moe_layer(g, T, H, I, E, b1, b2, bs, act, with_zp=zp, skew=True)
    b1v, b2v = wl.normal(g, (E, 2 * I), act), wl.normal(g, (E, H), act)
    y = run_qmoe_ex(d, T, H, I, E, k, b1, b2, bs, act, layout, b1v, b2v, None, "f32", x_offset)
    ref = oracle.qmoe_ex(d["X"], act, d["logits"], "f32", k, True, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], b1v, b1,
                         d["fc2_w"], d["fc2_scales"], d["fc2_zp"], b2v, b2, I, bs, layout, threads=THREADS)
    check(y, ref, act, 1)  # CUDA cores: the elementwise rule


@pytest.mark.parametrize("T,E,k,layout", [(4, 1024, 8, "concat"), (5, 300, 6, "interleaved"), (3, 8, 1, "concat")])
def test_grouped_plan_router_sizes(T, E, k, layout):
    """The grouped CUDA-core plan from three tokens on: the largest router (E = 1024,
    one-CTA permutation with its m-tiles), an E that is not a power of two, and a
    single expert per token."""
    H, I, bs = 256, 128, 32
    g = wl.rng(seed("grouped-router", T, E, k, layout))
    d = wl.moe_layer(g, T, H, I, E, 3, 3, bs, "bf16", with_zp=True, skew=False)
    y = run_qmoe(d, T, H, I, E, k, 3, 3, bs, "bf16", layout)
    check(y, reference(d, k, 3, 3, I, bs, "bf16", layout), "bf16", 1)  # CUDA cores: the elementwise rule


@pytest.mark.parametrize("layout,H,bs", [("concat", 64, 32), ("concat", 96, 32)])
def test_tiled_plan_fallback(layout, H, bs):
    """Concatenated gate/up rows of less than 16 scale bytes with X rows off a
    16-byte boundary: the grouped plan cannot copy such row ranges, the tiled
    CUDA-core plan runs."""
    T, E, k, I = 20, 8, 2, 64
    g = wl.rng(seed("tiled-fallback", layout, H, bs))
    d = wl.moe_layer(g, T, H, I, E, 4, 3, bs, "f16", with_zp=True, skew=True)
    y = run_qmoe_ex(d, T, H, I, E, k, 4, 3, bs, "f16", layout, None, None, None, "f32", 1)
    ref = oracle.qmoe_ex(d["X"], "f16", d["logits"], "f32", k, True, d["fc1_w"], d["fc1_scales"], d["fc1_zp"], None, 4,
                         d["fc2_w"], d["fc2_scales"], d["fc2_zp"], None, 3, I, bs, layout, threads=THREADS)
    check(y, ref, "f16", 1)
