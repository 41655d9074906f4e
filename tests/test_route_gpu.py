"""GPU parity of routing (indices bit-exact, weights fp32 tolerance), the
expert-sorted permutation (bit-exact) and the raw-code unpack (bit-exact)."""
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


def seed(*key):
    return zlib.crc32(repr(key).encode())


def gpu_route(logits, k, normalize):
    T, E = logits.shape
    L = to_dev(logits)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    mnb.qmoe_route(L, k, normalize, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,E,k,skew", [(1, 128, 8, False), (1000, 128, 8, False), (4096, 128, 8, True),
                                        (257, 100, 7, False), (64, 64, 64, False), (33, 256, 40, False),
                                        (5, 1024, 3, False), (9, 1, 1, False), (17, 33, 32, True)])
@pytest.mark.parametrize("normalize", [True, False])
def test_route_matches_oracle(T, E, k, skew, normalize):
    g = wl.rng(seed("route", T, E, k, skew))
    logits = wl.router_logits(g, T, E, skew)
    idx, w = gpu_route(logits, k, normalize)
    ridx, rw = oracle.route(logits, k, normalize)
    assert np.array_equal(idx, ridx)
    assert_f32_close(w, rw)


def test_route_ties_and_equal_logits():
    g = wl.rng(seed("ties"))
    logits = np.round(g.standard_normal((300, 128)) * 1.5).astype(np.float32)  # heavy ties
    logits[0] = 0.0
    logits[1, :] = -0.0
    logits[1, 77] = 0.0
    for k in (1, 8, 31):
        idx, w = gpu_route(logits, k, True)
        ridx, rw = oracle.route(logits, k, True)
        assert np.array_equal(idx, ridx)
        assert_f32_close(w, rw)
    idx, w = gpu_route(logits[:1], 8, True)
    assert idx[0].tolist() == list(range(8)) and np.all(w == np.float32(1 / 8))


@pytest.mark.parametrize("T,k,E,skew", [(1, 8, 128, False), (4096, 8, 128, True), (513, 8, 128, False),
                                        (100, 3, 1000, False), (2048, 1, 7, True), (31, 32, 64, False)])
def test_permute_matches_oracle(T, k, E, skew):
    g = wl.rng(seed("perm", T, k, E))
    ridx, _ = oracle.route(wl.router_logits(g, T, E, skew), k, True)
    idx = to_dev(ridx)
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    mnb.qmoe_permute(idx, E, counts, offsets, perm)
    c, o, p = oracle.permute(ridx, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(perm.cpu().numpy(), p)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("K", [2048, 2080, 77])
def test_unpack_codes_bit_exact(bits, bs, K):
    g = wl.rng(seed("unpack", bits, bs, K))
    rows = 37
    packed = wl.random_bytes(g, (rows, oracle.row_bytes(K, bits, bs)))
    codes = torch.zeros((rows, K), dtype=torch.uint8, device="cuda")
    mnb.mnb_unpack_codes(to_dev(packed), rows, K, bits, bs, codes)
    assert np.array_equal(codes.cpu().numpy(), oracle.unpack_codes(packed, rows, K, bits, bs))


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("bs", [32, 64, 128])
def test_pack_and_unpack_every_width(bits, bs):
    """Row-local LSB-first packing for widths 1..8 ("P0: Portable Format"):
    the GPU pack equals the oracle's bytes (zero padding in a partial last
    block, code bits above the width ignored) and the GPU unpack returns the
    codes."""
    g = wl.rng(zlib.crc32(repr(("pack", bits, bs)).encode()))
    rows, K = 37, 3 * bs + 11
    codes = g.integers(0, 256, size=(rows, K), dtype=np.uint8)
    ref = oracle.pack_codes(codes & ((1 << bits) - 1), bits, bs)
    packed = torch.empty(ref.shape, dtype=torch.uint8, device="cuda")
    mnb.mnb_pack_codes(to_dev(codes), rows, K, bits, bs, packed)
    got = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    mnb.mnb_unpack_codes(packed, rows, K, bits, bs, got)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), ref)
    assert np.array_equal(got.cpu().numpy(), codes & ((1 << bits) - 1))
