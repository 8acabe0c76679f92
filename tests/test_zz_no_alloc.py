"""fp8_linear_noalloc: the linear for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: code hosted inside an application that
owns all device memory and passes a kernel only its inputs and outputs, or a latency-
critical path that must not call cudaMalloc (it can wait for other device work). For them
the library keeps its scratch in one fixed array per GPU. These tests call that entry point
through the C ABI and compare it with fp8_linear / fp8_linear_channelwise, which use a
caller workspace, on two calls in a row (the array keeps the previous call's contents).

This file is named so that pytest collects it after every other test file.
"""

import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from oracle import fp8_oracle as O
from parity import f32, oracle_act, oracle_weight

DEV = "cuda:0"


@pytest.fixture(scope="module")
def L():
    _build.build()
    return F.lib()


def call_noalloc(L, a, qw, s_w, per_channel, bias, y):
    """Direct C-ABI call; returns the status code."""
    stream = torch.cuda.current_stream(a.device).cuda_stream
    return L.fp8_linear_noalloc(a.data_ptr(), a.shape[0], a.shape[1], a.stride(0), qw.data_ptr(), qw.shape[0],
                                qw.stride(0), s_w.data_ptr(), int(per_channel),
                                None if bias is None else bias.data_ptr(), y.data_ptr(), y.stride(0), stream)


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,N,per_channel", [(7, 2050, 3001, False),    # decode GEMV path
                                               (15, 4096, 4096, True),
                                               (24, 4096, 2048, True),    # GEMV on A quantized first
                                               (300, 4100, 1027, True),   # tcgen05 GEMM path
                                               (1900, 4096, 768, False)])  # near the scratch limit
def test_noalloc_matches_workspace_entry_point(L, M, K, N, per_channel):
    assert F.min_workspace_bytes(M, K, N) <= F.FP8_NOALLOC_SCRATCH_BYTES
    w = I.weights_row_std(N, K, (930, M, N))
    bias = I.bias_normal(N, (931, N))
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=per_channel)
    b = bias.to(DEV)
    ref_fn = F.fp8_linear_channelwise if per_channel else F.fp8_linear
    ws_same = torch.empty(F.FP8_NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device=DEV)
    for call in range(2):  # second call reuses the scratch the first one left behind
        a = I.activations_heavy_tail(M, K, (932, M, call))
        ad = a.to(DEV)
        # the workspace entry point with a workspace of the scratch array's size plans the
        # same launches (the K split depends on the space available)
        y_ref = ref_fn(ad, qw, s_w, b, ws=ws_same)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert call_noalloc(L, ad, qw, s_w, per_channel, b, y) == F.FP8_OK
        torch.cuda.synchronize()
        assert F.fp8_last_device_status() == F.FP8_OK
        # tolerance of the parity tests, from the oracle's quantization of the same inputs
        # the same kernels on the same inputs: identical bits to the workspace entry point
        assert torch.equal(y, y_ref), f"call {call}: differs from the workspace entry point"
        # and within the parity tolerance of the oracle on the same seeded inputs
        qa_o, s_a_o = oracle_act(a)
        qw_o, s_w_o = oracle_weight(w, per_channel)
        y_o = O.scaled_mm(qa_o, s_a_o, qw_o, s_w_o, f32(bias))
        tol = O.tolerance(qa_o, s_a_o, qw_o, s_w_o, y_o)
        diff = np.abs(f32(y).astype(np.float64) - y_o.astype(np.float64))
        assert np.all(diff <= tol), f"call {call}: max diff/tol against the oracle {np.nanmax(diff / tol)}"


@pytest.mark.gpu
def test_noalloc_refuses_shapes_beyond_its_scratch(L):
    M, K, N = 4096, 4096, 256  # GEMM path: qA alone is 16 MiB
    a = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    qw = torch.zeros((N, K), dtype=torch.uint8, device=DEV)
    s_w = torch.ones(1, device=DEV)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    assert call_noalloc(L, a, qw, s_w, 0, None, y) == F.FP8_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not y.any()


def test_noalloc_rejects_bad_arguments_without_a_gpu(L):
    P = 0x7F0000000000
    f = L.fp8_linear_noalloc
    assert f(P, 4, 64, 64, P, 32, 64, P, 2, None, P, 32, None) == F.FP8_ERR_INVALID_ARG   # bad flag
    assert f(None, 4, 64, 64, P, 32, 64, P, 0, None, P, 32, None) == F.FP8_ERR_INVALID_ARG
    assert f(P, 4096, 4096, 4096, P, 32, 4096, P, 0, None, P, 32, None) == F.FP8_ERR_WORKSPACE
    assert f(P, 0, 64, 64, P, 32, 64, P, 0, None, P, 32, None) == F.FP8_OK
