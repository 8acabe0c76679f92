"""The decode GEMV at 17 to 32 tokens (four n8 token tiles, main loop on tcgen05), with the
crossover raised to 32: parity against the oracle for every path (bf16 activations quantized
once, dynamic or static, then loaded by TMA; pre-quantized activations; weight-only bf16
activations) and both FP8 formats."""

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from oracle import fp8_oracle as O
from parity import (assert_guards_intact, f32, guarded, linear_parity, oracle_weight, weight_only_parity)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def gemv_through_32():
    _build.build()
    F.lib()
    prev = F.fp8_set_gemv_max_m(32)
    assert F.fp8_set_gemv_max_m(-1) == 32
    yield
    F.fp8_set_gemv_max_m(prev)


def linear(a, qw, s_w, per_channel, bias=None, **kw):
    """The linear into a guarded output; returns Y after checking the guard bands and status."""
    M, N = a.shape[0], qw.shape[0]
    buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
    F.fp8_linear_ex(a, qw, s_w, per_channel=per_channel, bias=bias, out=y, **kw)
    torch.cuda.synchronize()
    assert_guards_intact(buf, base, row_bytes, used, M)
    assert F.fp8_last_device_status() == F.FP8_OK
    return y


@pytest.mark.parametrize("M", [17, 20, 24, 25, 31, 32])
def test_gemv_wide_every_m(M):
    K, N = 1000, 1027
    assert F.fp8_uses_gemv(M, K, N) and F.fp8_workspace_bytes(M, K, N) == F.min_workspace_bytes(M, K, N) > 0
    a = I.activations_normal(M, K, (940, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (941,))
    b = I.bias_normal(N, (942,))
    for pc in (False, True):
        qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=pc)
        y = linear(a.to(DEV), qw, s_w, pc, b.to(DEV))
        linear_parity(y, a, w, pc, b, what=f"gemv M={M} pc={pc}")


@pytest.mark.parametrize("layer", range(4))
@pytest.mark.parametrize("M", [24, 32])
def test_gemv_wide_decode_layers(layer, M):
    """Mistral-7B linears at full size; Y on all rows and 1024 sampled columns."""
    L = I.LLAMA8B_LAYERS[layer]
    w = I.decode_weight(layer)
    a = I.decode_activations(M, layer)
    cols = np.unique(np.r_[np.random.default_rng(layer + 50).choice(L.N, 1024, replace=False), 0, L.N - 1])
    qw, s_w = F.fp8_quantize_weight(w.to(DEV))
    y = linear(a.to(DEV), qw, s_w, False)
    linear_parity(y, a, w, False, cols=cols, what=f"decode {L.name} M={M}")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("K", [4096, 8192])
def test_gemv_wide_in_kernel_codes(fmt, static, K):
    """W = I at M = 32: each output is one product, so every code the quantizer chose (before the
    GEMV) and the GEMV's use of it are checked."""
    M = 32
    g = np.random.default_rng(943 + K)
    a = I.to_bf16((g.standard_normal((M, K)) * np.exp2(g.integers(-14, 9, (M, K)))).astype(np.float32))
    w = torch.eye(K, dtype=torch.bfloat16)
    s = np.float32(float(O.amax(f32(a))) / O.fp8_max(fmt) / 2) if static else None
    qw, s_w = F.fp8_quantize_weight(w.to(DEV))
    s_dev = None if s is None else torch.tensor([s], dtype=torch.float32, device=DEV)
    y = linear(a.to(DEV), qw, s_w, False, fmt_a=fmt, s_static=s_dev)
    cols = np.sort(g.choice(K, 600, replace=False))
    linear_parity(y, a, w, False, cols=cols, what=f"identity {fmt} static={static}", fmt_a=fmt, s_static=s)


@pytest.mark.parametrize("fmt_a,fmt_w", [("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e5m2", "e5m2")])
def test_gemv_wide_formats(fmt_a, fmt_w):
    M, K, N = 29, 2050, 3001
    a = I.activations_normal(M, K, (944,), outlier_cols=4)
    w = I.weights_row_std(N, K, (945,))
    qw, s_w = F.fp8_quantize_weight_ex(w.to(DEV), fmt_w, per_channel=True)
    y = linear(a.to(DEV), qw, s_w, True, fmt_a=fmt_a, fmt_w=fmt_w)
    linear_parity(y, a, w, True, what=f"formats {fmt_a}x{fmt_w}", fmt_a=fmt_a, fmt_w=fmt_w)


@pytest.mark.parametrize("M", [17, 32])
def test_gemv_wide_prequantized_equals_linear(M):
    """fp8_scaled_mm (pre-quantized activations) and fp8_linear (A quantized once, then the same
    GEMV) run the same MMAs in the same order: identical bits."""
    K, N = 4096, 777
    a = I.activations_normal(M, K, (946, M)).to(DEV)
    qw, s_w = F.fp8_quantize_weight(I.weights_row_std(N, K, (947,)).to(DEV), per_channel=True)
    y1 = F.fp8_linear_channelwise(a, qw, s_w)
    qa, s_a = F.fp8_quantize_act(a)
    y2 = F.fp8_scaled_mm(qa, K, s_a, qw, s_w, per_channel=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [17, 32])
def test_gemv_wide_weight_only(fmt, M):
    K, N = 1000, 1027
    assert F.fp8_weight_only_workspace_bytes(M, K, N) == 0
    a = I.activations_normal(M, K, (948, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (949,))
    b = I.bias_normal(N, (950,))
    for pc in (False, True):
        qw, s_w = F.fp8_quantize_weight_ex(w.to(DEV), fmt, per_channel=pc)
        buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
        F.fp8_linear_weight_only(a.to(DEV), qw, s_w, per_channel=pc, bias=b.to(DEV), out=y, fmt_w=fmt)
        torch.cuda.synchronize()
        assert_guards_intact(buf, base, row_bytes, used, M)
        assert F.fp8_last_device_status() == F.FP8_OK
        weight_only_parity(y, a, w, pc, b, what=f"wo gemv M={M} {fmt} pc={pc}", fmt_w=fmt)


def test_crossover_setter_clamps():
    prev = F.fp8_set_gemv_max_m(100)
    assert F.fp8_set_gemv_max_m(-1) == 32
    F.fp8_set_gemv_max_m(0)
    assert not F.fp8_uses_gemv(1, 4096, 4096)
    F.fp8_set_gemv_max_m(prev)
    assert F.fp8_uses_gemv(32, 4096, 4096)
