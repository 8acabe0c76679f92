"""Failure detection without a GPU fault: the library's bounded device waits give up after a
limit, record an error word that fp8_last_device_status turns into FP8_ERR_TIMEOUT, and the
context stays usable. The self-test kernel withholds one item from its consumer (a flag that
nothing sets); nothing faults, traps or hangs."""

import time

import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from parity import linear_parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    F.lib()


def test_bounded_wait_runs_out_and_is_reported_once():
    torch.cuda.synchronize()
    assert F.fp8_last_device_status() == F.FP8_OK  # nothing pending
    limit_ns = 30_000_000
    t0 = time.perf_counter()
    assert F.fp8_selftest_timeout(limit_ns) == F.FP8_OK
    assert F.fp8_last_device_status() == F.FP8_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert limit_ns * 1e-9 <= elapsed < 5.0, elapsed  # the wait ran out, it did not hang
    assert F.fp8_last_device_status() == F.FP8_OK     # reported once, then cleared


def test_context_is_usable_after_a_timeout():
    assert F.fp8_selftest_timeout(5_000_000) == F.FP8_OK
    assert F.fp8_last_device_status() == F.FP8_ERR_TIMEOUT
    for M in (3, 100):  # decode GEMV and tcgen05 GEMM paths
        a = I.activations_normal(M, 1024, (501, M))
        w = I.weights_normal(512, 1024, (502,))
        qw, s_w = F.fp8_quantize_weight(w.to(DEV))
        y = F.fp8_linear(a.to(DEV), qw, s_w)
        torch.cuda.synchronize()
        assert F.fp8_last_device_status() == F.FP8_OK
        linear_parity(y, a, w, False, what=f"after timeout M={M}")
