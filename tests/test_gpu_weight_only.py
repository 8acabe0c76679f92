"""GPU parity of the weight-only FP8 linear (bf16 activations, FP8 weights up-converted to bf16)
against the oracle: the decode GEMV path (tiles up-converted in registers, bf16 MMAs) and the
GEMM path (up-conversion pass + tcgen05 kind::f16 GEMM)."""

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from oracle import fp8_oracle as O
from parity import (assert_codes_equal, assert_guards_intact, assert_scale_equal, f32, guarded, oracle_weight,
                    tail_rows, weight_only_parity)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    F.lib()


def run_wo(a_cpu, w_cpu, fmt_w, per_channel, bias_cpu=None, lda_pad=0, check_w=True):
    M, K = a_cpu.shape
    N = w_cpu.shape[0]
    qw, s_w = F.fp8_quantize_weight_ex(w_cpu.to(DEV), fmt_w, per_channel=per_channel)
    if lda_pad:
        big = torch.zeros((M, K + lda_pad), dtype=torch.bfloat16)
        big[:, :K] = a_cpu
        a = big.to(DEV)[:, :K]
    else:
        a = a_cpu.to(DEV)
    buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
    F.fp8_linear_weight_only(a, qw, s_w, per_channel=per_channel,
                             bias=None if bias_cpu is None else bias_cpu.to(DEV), out=y, fmt_w=fmt_w)
    torch.cuda.synchronize()
    assert_guards_intact(buf, base, row_bytes, used, M)
    assert F.fp8_last_device_status() == F.FP8_OK
    if check_w:
        q_ref, s_ref = oracle_weight(w_cpu, per_channel, fmt=fmt_w)
        assert_scale_equal(s_w, s_ref, f"s_w {fmt_w}")
        assert_codes_equal(qw, q_ref, K, f"qW {fmt_w}")
    return y


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16])
def test_weight_only_decode(fmt, M):
    K, N = 1000, 1027
    assert F.fp8_weight_only_workspace_bytes(M, K, N) == 0
    a = I.activations_normal(M, K, (301, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (302,))
    b = I.bias_normal(N, (303,))
    for per_channel in (False, True):
        y = run_wo(a, w, fmt, per_channel, b)
        weight_only_parity(y, a, w, per_channel, b, what=f"wo gemv M={M} {fmt} pc={per_channel}", fmt_w=fmt)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("K", [4096, 14336, 16384, 32768])
def test_weight_only_decode_layer_k(fmt, K):
    for M in (1, 16):
        N = 1500
        a = I.activations_normal(M, K, (304, M, K))
        w = I.weights_row_std(N, K, (305, K))
        y = run_wo(a, w, fmt, True, lda_pad=8 if M == 16 else 0)
        weight_only_parity(y, a, w, True, what=f"wo gemv M={M} K={K} {fmt}", fmt_w=fmt)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,K,N,pad", [(40, 1000, 1027, 0), (300, 2048, 640, 0), (129, 1001, 700, 0),
                                       (200, 1024, 513, 3), (5, 32800, 300, 0)])
def test_weight_only_gemm(fmt, M, K, N, pad):
    """GEMM path: ragged M, N and K, K not a multiple of 8 and an odd row stride (A is copied to an
    aligned buffer), and a decode-sized M whose K is beyond the GEMV's slice budget."""
    assert F.fp8_weight_only_workspace_bytes(M, K, N) > 0
    a = I.activations_heavy_tail(M, K, (306, M, K))
    w = I.weights_row_std(N, K, (307, N, K))
    b = I.bias_normal(N, (308, N))
    for per_channel in (False, True):
        y = run_wo(a, w, fmt, per_channel, b, lda_pad=pad)
        weight_only_parity(y, a, w, per_channel, b, what=f"wo gemm {M}x{K}x{N} {fmt} pc={per_channel}",
                           fmt_w=fmt)


@pytest.mark.parametrize("M", [1, 16, 64])
@pytest.mark.parametrize("fmt,one", [("e4m3", 0x38), ("e5m2", 0x3C)])
def test_weight_only_identity_weights_are_exact(M, fmt, one):
    """qW = I (the code of 1.0) with s_w = 0.75: every output is the single exact product
    bf16(0.75 * a), so the up-conversion and the scale are checked bit for bit."""
    K = 2048
    g = np.random.default_rng(309 + M)
    a = I.to_bf16((g.standard_normal((M, K)) * np.exp2(g.integers(-30, 30, (M, K)))).astype(np.float32))
    qw = torch.zeros((K, K), dtype=torch.uint8)
    qw[torch.arange(K), torch.arange(K)] = one
    s_w = torch.tensor([0.75], dtype=torch.float32, device=DEV)
    ws_need = F.fp8_weight_only_workspace_bytes(M, K, K)
    y = F.fp8_linear_weight_only(a.to(DEV), qw.to(DEV), s_w, fmt_w=fmt)
    torch.cuda.synchronize()
    want = O.bf16_round(f32(a).astype(np.float64) * 0.75)
    assert np.array_equal(f32(y), want), f"M={M} {fmt} ws={ws_need}"


def test_weight_only_prefill_sampled():
    """Llama-3-8B gate_up at M = 4096 on the GEMM path, 24 sampled rows x all columns."""
    L = I.LLAMA8B_LAYERS[2]
    M = 4096
    a = I.prefill_activations(2, M=M)
    w = I.prefill_weight(2)
    y = run_wo(a, w, "e4m3", True, check_w=False)
    rows = np.sort(np.random.default_rng(310).choice(M, 24, replace=False))
    weight_only_parity(y, a, w, True, rows=rows, what=f"wo prefill {L.name}")


def test_weight_only_tail_split():
    """bf16 kernel (kind::f16) with the last, partial wave split by columns into 128-column units
    over all of K: ragged M, N and K against the oracle, both scale modes."""
    K, N = 520, 2500
    qa0 = torch.zeros((4096, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    qw0 = torch.zeros((N, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    cfg0 = F.fp8_gemm_config(qa0, qw0, K)  # the same tile grid and slots as the bf16 kernel
    assert cfg0["two_sm"]
    M = tail_rows((N + 255) // 256, cfg0["grid"] // 2, 2, 256)
    assert F.fp8_gemm_config(qa0[:M], qw0, K)["tail_split"] == 2
    a = I.activations_heavy_tail(M, K, (311, M))
    w = I.weights_row_std(N, K, (312, N))
    b = I.bias_normal(N, (313, N))
    for per_channel in (False, True):
        y = run_wo(a, w, "e4m3", per_channel, b, check_w=False)
        weight_only_parity(y, a, w, per_channel, b, what=f"wo tail {M}x{K}x{N} pc={per_channel}")


def test_weight_only_matches_scaled_bf16_product_of_upconverted_weights():
    """GPU against GPU: the weight-only Y equals bf16(s_w * (A @ decode(qW)^T)) computed by torch in
    fp32 on the same device within the tolerance (a check independent of the oracle)."""
    M, K, N = 64, 1024, 512
    a = I.activations_normal(M, K, (311,)).to(DEV)
    qw, s_w = F.fp8_quantize_weight(I.weights_normal(N, K, (312,)).to(DEV), per_channel=True)
    y = F.fp8_linear_weight_only(a, qw, s_w, per_channel=True)
    wdec = qw[:, :K].view(torch.float8_e4m3fn).float()
    ref = ((a.float() @ wdec.t()) * s_w[None, :]).bfloat16()
    torch.cuda.synchronize()
    err = (y.float() - ref.float()).abs()
    tol = ref.float().abs() * 2.0 ** -7 + K * 2.0 ** -23 * (a.float().abs() @ (wdec.abs() * s_w[:, None]).t())
    assert bool((err <= tol).all())
