"""CPU-side checks of the C ABI: the library builds and loads, it exports every
function include/mnb.h declares, and every metadata error is reported before
any GPU work (these calls return before touching CUDA, so they run without a
GPU).  Also the host content validator."""
import ctypes
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl
from qmoe_mnb_matmul_gb300 import _build
import qmoe_mnb_matmul_gb300 as mnb

OK, INVALID, UNSUPPORTED, OVERFLOW, WORKSPACE, CONTENT = 0, 1, 2, 3, 4, 7


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mnb.load_library()


def test_exports_every_declared_symbol(lib):
    names = mnb.header_functions()
    assert len(names) >= 10
    dyn = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in dyn.splitlines() if " T " in line}
    for n in names:
        assert n in exported, f"{n} is declared in include/mnb.h but not exported"
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    for code, name in mnb._binding.STATUS.items():
        assert mnb.mnb_status_string(code) == name
    assert mnb.mnb_status_string(99) == "MNB_ERR_UNKNOWN"


FAKE = 0x10000  # 64 KiB-aligned fake device address: never dereferenced by these calls


def call_matmul(lib, A=FAKE, a_dt=0, M=1, K=256, B=FAKE, S=FAKE, s_dt=0, Z=None, N=128, bits=4, bs=32, Y=FAKE,
                y_dt=0):
    return lib.mnb_matmul(A, a_dt, M, K, B, S, s_dt, Z, N, bits, bs, Y, y_dt, None, 0, None)


def test_matmul_metadata_errors(lib):
    assert call_matmul(lib, A=None) == INVALID
    assert call_matmul(lib, B=None) == INVALID
    assert call_matmul(lib, S=None) == INVALID
    assert call_matmul(lib, Y=None) == INVALID
    assert call_matmul(lib, M=0) == INVALID
    assert call_matmul(lib, K=0) == INVALID
    assert call_matmul(lib, N=-1) == INVALID
    assert call_matmul(lib, a_dt=7) == INVALID
    assert call_matmul(lib, bits=9) == UNSUPPORTED   # widths 1..8 only
    assert call_matmul(lib, bits=0) == UNSUPPORTED
    assert call_matmul(lib, bs=16) == UNSUPPORTED
    assert call_matmul(lib, bs=256) == UNSUPPORTED
    assert call_matmul(lib, a_dt=1, s_dt=2) == UNSUPPORTED  # scale dtype must be f32 or the activation dtype
    assert call_matmul(lib, B=FAKE + 8) == UNSUPPORTED       # packed weights must be 16-byte aligned
    assert call_matmul(lib, S=FAKE + 4) == UNSUPPORTED
    assert call_matmul(lib, A=FAKE + 2) == UNSUPPORTED       # fp32 activations must be 4-byte aligned
    assert call_matmul(lib, N=1 << 40, K=1 << 30) == OVERFLOW


def test_workspace_size_queries(lib):
    n = ctypes.c_size_t(123)
    assert lib.mnb_matmul_workspace_size(1, 2048, 4096, 4, 32, 0, ctypes.byref(n)) == OK
    assert n.value == 0
    assert lib.mnb_matmul_workspace_size(1, 2048, 4096, 4, 32, 0, None) == INVALID
    assert lib.mnb_matmul_workspace_size(1, 2048, 4096, 9, 32, 0, ctypes.byref(n)) == UNSUPPORTED
    assert lib.mnb_matmul_workspace_size(64, 2048, 4096, 6, 32, 1, ctypes.byref(n)) == OK  # CUDA cores: none
    assert n.value == 0
    assert lib.qmoe_workspace_size(1, 2048, 768, 128, 8, 1, ctypes.byref(n)) == OK
    assert n.value > 0
    small = n.value
    assert lib.qmoe_workspace_size(4096, 2048, 768, 128, 8, 1, ctypes.byref(n)) == OK
    assert n.value >= small
    assert lib.qmoe_workspace_size(1, 2048, 768, 128, 200, 1, ctypes.byref(n)) == INVALID   # k > E
    assert lib.qmoe_workspace_size(1, 2048, 768, 128, 8, 0, ctypes.byref(n)) == UNSUPPORTED  # fp32 activations


def call_qmoe(lib, X=FAKE, act=1, T=1, H=2048, L=FAKE, E=128, k=8, W1=FAKE, S1=FAKE, b1=3, W2=FAKE, S2=FAKE, b2=3,
              I=768, bs=64, layout=0, Y=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return lib.qmoe_forward(X, act, T, H, L, E, k, 1, W1, S1, None, b1, W2, S2, None, b2, I, bs, layout, Y, ws,
                            ws_bytes, None)


def test_qmoe_metadata_errors(lib):
    assert call_qmoe(lib, X=None) == INVALID
    assert call_qmoe(lib, L=None) == INVALID
    assert call_qmoe(lib, k=0) == INVALID
    assert call_qmoe(lib, k=129) == INVALID
    assert call_qmoe(lib, layout=2) == INVALID
    assert call_qmoe(lib, act=0) == UNSUPPORTED            # QMoE activations are f16 / bf16
    assert call_qmoe(lib, b1=2) == UNSUPPORTED
    assert call_qmoe(lib, H=2047) == UNSUPPORTED           # H must be a multiple of the block size
    assert call_qmoe(lib, I=700) == UNSUPPORTED            # and so must I
    assert call_qmoe(lib, E=2000, k=8) == UNSUPPORTED
    assert call_qmoe(lib, W1=FAKE + 4) == UNSUPPORTED
    assert call_qmoe(lib, ws=None) == WORKSPACE
    assert call_qmoe(lib, ws_bytes=16) == WORKSPACE


def test_route_permute_unpack_metadata_errors(lib):
    assert lib.qmoe_route(None, 1, 128, 8, 1, FAKE, FAKE, None) == INVALID
    assert lib.qmoe_route(FAKE, 1, 128, 129, 1, FAKE, FAKE, None) == INVALID
    assert lib.qmoe_route(FAKE, 1, 2048, 8, 1, FAKE, FAKE, None) == UNSUPPORTED
    assert lib.qmoe_permute(FAKE, 0, 8, 128, FAKE, FAKE, FAKE, None) == INVALID
    assert lib.qmoe_permute(FAKE, 1 << 30, 8, 128, FAKE, FAKE, FAKE, None) == OVERFLOW
    assert lib.mnb_unpack_codes(FAKE, 4, 64, 9, 32, FAKE, None) == UNSUPPORTED   # widths 1..8
    assert lib.mnb_unpack_codes(FAKE, 4, 64, 0, 32, FAKE, None) == UNSUPPORTED
    assert lib.mnb_unpack_codes(FAKE, 4, 64, 5, 16, FAKE, None) == UNSUPPORTED
    assert lib.mnb_unpack_codes(None, 4, 64, 4, 32, FAKE, None) == INVALID
    assert lib.mnb_pack_codes(None, 4, 64, 4, 32, FAKE, None) == INVALID
    assert lib.mnb_pack_codes(FAKE, 0, 64, 4, 32, FAKE, None) == INVALID
    assert lib.mnb_pack_codes(FAKE, 4, 64, 9, 32, FAKE, None) == UNSUPPORTED
    assert lib.mnb_pack_codes(FAKE, 4, 64, 6, 48, FAKE, None) == UNSUPPORTED
    assert lib.mnb_pack_codes(FAKE, 1 << 40, 1 << 30, 8, 32, FAKE, None) == OVERFLOW


def test_quantize_int3_metadata_errors(lib):
    q = lib.mnb_quantize_int3
    assert q(None, 0, 4, 64, 32, FAKE, FAKE, 1, None) == INVALID
    assert q(FAKE, 0, 4, 64, 32, None, FAKE, 1, None) == INVALID
    assert q(FAKE, 0, 0, 64, 32, FAKE, FAKE, 1, None) == INVALID
    assert q(FAKE, 3, 4, 64, 32, FAKE, FAKE, 1, None) == INVALID       # no such dtype
    assert q(FAKE, 0, 4, 64, 48, FAKE, FAKE, 1, None) == UNSUPPORTED   # block size
    assert q(FAKE, 0, 4, 80, 32, FAKE, FAKE, 1, None) == UNSUPPORTED   # K not a multiple of the block
    assert q(FAKE + 4, 0, 4, 64, 32, FAKE, FAKE, 1, None) == INVALID   # W not 16-byte aligned
    assert q(FAKE, 0, 4, 64, 32, FAKE + 2, FAKE, 1, None) == INVALID   # B_packed not 4-byte aligned
    assert q(FAKE, 0, 1 << 40, 1 << 30, 32, FAKE, FAKE, 1, None) == OVERFLOW


# ------------------------------------------------------- host validator

@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("bs", [32, 64, 128])
def test_validate_host_accepts_canonical_content(lib, bits, bs):
    g = wl.rng(3)
    N, K = 7, 2 * bs + 9  # partial last block -> padding bits
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    nb = oracle.n_blocks(K, bs)
    zp = oracle.pack_zero_points(g.integers(0, 1 << bits, size=(N, nb), dtype=np.uint8), bits)
    scales = wl.uniform(g, (N, nb), 0.005, 0.02, "f16")
    assert mnb.mnb_validate_host(packed, scales, 1, zp, N, K, bits, bs) == OK
    assert mnb.mnb_validate_host(packed, scales, 1, None, N, K, bits, bs) == OK


def test_validate_host_rejects_malformed_content(lib):
    g = wl.rng(4)
    N, K, bits, bs = 5, 100, 3, 32
    codes = g.integers(0, 8, size=(N, K), dtype=np.uint8)
    packed = oracle.pack_codes(codes, bits, bs)
    nb = oracle.n_blocks(K, bs)
    scales = np.full((N, nb), 0.01, np.float32)
    zp = oracle.pack_zero_points(np.full((N, nb), 4, np.uint8), bits)
    assert mnb.mnb_validate_host(packed, scales, 0, zp, N, K, bits, bs) == OK
    bad = packed.copy()
    bad[2, -1] |= 0x80  # a padding bit of row 2
    assert mnb.mnb_validate_host(bad, scales, 0, zp, N, K, bits, bs) == CONTENT
    badz = zp.copy()
    badz[1, -1] |= 0x80  # 4 blocks * 3 bits = 12 bits -> bits 12..15 of the 2-byte row are padding
    assert mnb.mnb_validate_host(packed, scales, 0, badz, N, K, bits, bs) == CONTENT
    for v in (np.nan, np.inf, -0.5):
        s = scales.copy()
        s[3, 1] = v
        assert mnb.mnb_validate_host(packed, s, 0, zp, N, K, bits, bs) == CONTENT
    s = scales.copy()
    s[0, 0] = -0.0  # negative zero is not negative
    assert mnb.mnb_validate_host(packed, s, 0, zp, N, K, bits, bs) == OK
    h = wl.cast(scales, "bf16")
    h[4, 2] = 0x7F80  # bf16 +inf
    assert mnb.mnb_validate_host(packed, h, 2, zp, N, K, bits, bs) == CONTENT
    h = wl.cast(scales, "f16")
    h[0, 3] = 0xBC00  # f16 -1.0
    assert mnb.mnb_validate_host(packed, h, 1, zp, N, K, bits, bs) == CONTENT
