"""Failure detection on the GPU without a fault: a kernel whose bounded wait runs
out (an mbarrier nothing arrives at, no copy, tensor-core operation or tensor
memory in flight) records MNB_ERR_TIMEOUT in the device error word and returns;
the error word reports it once, and the library keeps computing correct results
afterwards on the same context."""
import os
import time
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests._util import assert_close, assert_f32_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import qmoe_mnb_matmul_gb300 as mnb  # noqa: E402

THREADS = os.cpu_count() or 1
TIMEOUT = 6  # MNB_ERR_TIMEOUT


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    assert mnb.mnb_get_last_device_error() == 0
    t0 = time.perf_counter()
    mnb.mnb_diag_wait_timeout(2_000_000)  # 2 ms
    assert mnb.mnb_get_last_device_error() == TIMEOUT
    assert time.perf_counter() - t0 >= 2e-3
    assert mnb.mnb_get_last_device_error() == 0  # reported once, then cleared

    g = wl.rng(zlib.crc32(b"after-timeout"))
    # the decode GEMV (CUDA cores) and a tensor-core GEMM on the same context
    for M, a_dt, y_dt in ((1, "f32", "f32"), (64, "f16", "f16")):
        K, N = 2048, 1024
        packed, scales, _ = wl.quantized_weight(g, N, K, 4, 32)
        A = wl.normal(g, (M, K), a_dt)
        Y = torch.empty((M, N), dtype=getattr(torch, {"f32": "float32", "f16": "float16"}[y_dt]), device="cuda")
        mnb.mnb_matmul(to_dev(A, a_dt), to_dev(packed), to_dev(scales), None, N, 4, 32, Y, K=K, M=M)
        assert mnb.mnb_get_last_device_error() == 0
        ref = oracle.mnb_matmul(A, a_dt, packed, scales, "f32", None, N, K, 4, 32, threads=THREADS)
        assert_close(to_f64(Y), ref, y_dt, a_dt, tensor_cores=M >= 16)


def test_timeouts_on_two_streams_are_each_reported():
    s = torch.cuda.Stream()
    mnb.mnb_diag_wait_timeout(1_000_000, stream=s)
    assert mnb.mnb_get_last_device_error(s) == TIMEOUT
    mnb.mnb_diag_wait_timeout(1_000_000)
    assert mnb.mnb_get_last_device_error() == TIMEOUT
    assert mnb.mnb_get_last_device_error() == 0


def test_limits_outside_the_accepted_range_are_rejected():
    assert mnb.mnb_diag_wait_timeout(10, check=False) == 1          # below 1 us
    assert mnb.mnb_diag_wait_timeout(5_000_000_000, check=False) == 1  # above 1 s
    assert mnb.mnb_get_last_device_error() == 0
