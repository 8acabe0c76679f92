"""GPU parity of the wider rows: float8_e5m2 operands (any pairing with e4m3) and the static
(calibrated) activation scale, on the quantize kernels, the decode GEMV and the tcgen05 GEMM.

Codes and scales must be bit-exact against the oracle; Y within one bf16 ulp plus
K * 2^-23 * sum_k |a_k w_k| (oracle.tolerance for the formats in use).
"""

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from oracle import fp8_oracle as O
from parity import (assert_codes_equal, assert_guards_intact, assert_scale_equal, f32, guarded, linear_parity,
                    oracle_act, oracle_weight)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAIRS = [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")]


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    F.lib()


def all_finite_bf16() -> torch.Tensor:
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return bits[torch.isfinite(bits.float())]


def dev_scalar(v) -> torch.Tensor:
    return torch.tensor([float(np.float32(v))], dtype=torch.float32, device=DEV)


# --------------------------------------------------------------------------- quantization

@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("shape", [(256, 256), (3001, 2050), (1027, 1000)])
def test_e5m2_weight_quantization(per_channel, shape):
    N, K = shape
    w = I.weights_row_std(N, K, (177, N, K))
    qw, s_w = F.fp8_quantize_weight_ex(w.to(DEV), "e5m2", per_channel=per_channel)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_weight(w, per_channel, fmt="e5m2")
    assert_scale_equal(s_w, s_ref, f"e5m2 W {shape}")
    assert_codes_equal(qw, q_ref, K, f"e5m2 W {shape}")


def test_e5m2_all_bf16_values_under_many_scales():
    """Every finite bf16 value at 30 amax values (random, and 57344 * 2^k where quotients land
    on e5m2 rounding midpoints): dynamic e5m2 codes and scale bit-exact."""
    x = all_finite_bf16()
    g = np.random.default_rng(121)
    targets = [float(v) for v in g.standard_normal(20) * np.exp2(g.integers(-40, 40, 20))]
    targets += [57344.0 * 2.0 ** k for k in (-30, -16, -9, -3, -1, 0, 1, 5, 17, 60)]
    for T in targets:
        T = abs(float(torch.tensor(T).bfloat16().float()))
        v = x[x.float().abs() <= T]
        v = torch.cat([v, torch.tensor([T, -T], dtype=torch.bfloat16)])
        a = torch.cat([v, torch.zeros((-v.numel()) % 240, dtype=torch.bfloat16)]).view(-1, 240)
        qa, s_a = F.fp8_quantize_act_ex(a.to(DEV), "e5m2")
        torch.cuda.synchronize()
        q_ref, s_ref = oracle_act(a, fmt="e5m2")
        assert_scale_equal(s_a, s_ref, f"e5m2 amax {T:g}")
        assert_codes_equal(qa, q_ref, 240, f"e5m2 amax {T:g}")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("factor", [0.25, 1.0, 3.0])
def test_static_scale_quantization(fmt, factor):
    """A calibrated scale smaller than amax / max saturates the large elements; a larger one
    leaves headroom. Codes bit-exact; s_a receives a copy of the given scale."""
    a = I.activations_normal(97, 1000, (178,), outlier_cols=4)
    s = np.float32(float(O.amax(f32(a))) / O.fp8_max(fmt) * factor)
    qa, s_a = F.fp8_quantize_act_ex(a.to(DEV), fmt, s_static=dev_scalar(s))
    torch.cuda.synchronize()
    q_ref, _ = oracle_act(a, fmt=fmt, s_static=s)
    assert_scale_equal(s_a, s, f"static {fmt} x{factor}")
    assert_codes_equal(qa, q_ref, 1000, f"static {fmt} x{factor}")
    top = 0x7E if fmt == "e4m3" else 0x7B
    if factor < 1:
        assert np.any((qa.cpu().numpy()[:, :1000] & 0x7F) == top)


def test_static_scale_all_bf16_values():
    x = all_finite_bf16()
    a = torch.cat([x, torch.zeros((-x.numel()) % 255, dtype=torch.bfloat16)]).view(-1, 255)
    for fmt in ("e4m3", "e5m2"):
        for s in (1.0, 2.0 ** -20, 3.7e-3, 1.1e17):
            qa, _ = F.fp8_quantize_act_ex(a.to(DEV), fmt, s_static=dev_scalar(s))
            torch.cuda.synchronize()
            q_ref, _ = oracle_act(a, fmt=fmt, s_static=s)
            assert_codes_equal(qa, q_ref, 255, f"static {fmt} s={s:g} over all bf16")


def flat_rows(v: torch.Tensor, width: int = 256) -> torch.Tensor:
    """v padded with zeros into rows of `width` (a multiple of 16: ld == ldq == K, the
    gap-free layout the cast kernel streams without row arithmetic)."""
    return torch.cat([v, torch.zeros((-v.numel()) % width, dtype=torch.bfloat16)]).view(-1, width)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_static_scale_all_bf16_values_flat_rows(fmt):
    """Every finite bf16 value and +-inf in gap-free 256-wide rows, at scales inside, on the
    edges of and just outside the range where the cast computes x / s without division
    ([2^-80, 2^100]): codes bit-exact. The infinities and quotients beyond fp32 leave the
    branch-free path through its NaN-code check and saturate."""
    x = torch.cat([all_finite_bf16(), torch.tensor([float("inf"), float("-inf")], dtype=torch.bfloat16)])
    a = flat_rows(x)
    for s in (1.0, 2.0 ** -80, 2.0 ** -81, 2.0 ** 100, 2.0 ** 101, 3.7e-3, 1.1e17, 1e-30, 3.375 / 448, 0.5 / 448):
        s = float(np.float32(s))
        qa, _ = F.fp8_quantize_act_ex(a.to(DEV), fmt, s_static=dev_scalar(s))
        torch.cuda.synchronize()
        q_ref, _ = oracle_act(a, fmt=fmt, s_static=s)
        assert_codes_equal(qa, q_ref, 256, f"static {fmt} s={s:g} over all bf16, flat rows")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_dynamic_all_bf16_values_flat_rows(fmt):
    """Every finite bf16 value up to an amax, in gap-free rows, for amax values whose scale
    amax / max has few significant bits (mantissa a multiple of 7, or of 27, or a power of
    two: many quotients sit exactly on FP8 rounding midpoints) and random ones: dynamic codes
    and scale bit-exact."""
    x = all_finite_bf16()
    g = np.random.default_rng(122)
    targets = [float(v) for v in np.abs(g.standard_normal(8)) * np.exp2(g.integers(-30, 30, 8))]
    targets += [3.5, 3.375, 4.0, 7.0 * 2.0 ** -12, 27.0 * 2.0 ** 9, 1.0, O.fp8_max(fmt), 2.0 ** 70]
    for T in targets:
        T = abs(float(torch.tensor(T).bfloat16().float()))
        v = x[x.float().abs() <= T]
        a = flat_rows(torch.cat([v, torch.tensor([T, -T], dtype=torch.bfloat16)]))
        qa, s_a = F.fp8_quantize_act_ex(a.to(DEV), fmt)
        torch.cuda.synchronize()
        q_ref, s_ref = oracle_act(a, fmt=fmt)
        assert_scale_equal(s_a, s_ref, f"dynamic {fmt} amax {T:g}")
        assert_codes_equal(qa, q_ref, 256, f"dynamic {fmt} amax {T:g}, flat rows")


# --------------------------------------------------------------------------- linear

def run_ex(a_cpu, w_cpu, fmt_a, fmt_w, per_channel, bias_cpu=None, s_static=None, check_w=True):
    M, K = a_cpu.shape
    N = w_cpu.shape[0]
    qw, s_w = F.fp8_quantize_weight_ex(w_cpu.to(DEV), fmt_w, per_channel=per_channel)
    buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
    F.fp8_linear_ex(a_cpu.to(DEV), qw, s_w, per_channel=per_channel,
                    bias=None if bias_cpu is None else bias_cpu.to(DEV), out=y, fmt_a=fmt_a, fmt_w=fmt_w,
                    s_static=None if s_static is None else dev_scalar(s_static))
    torch.cuda.synchronize()
    assert_guards_intact(buf, base, row_bytes, used, M)
    assert F.fp8_last_device_status() == F.FP8_OK
    if check_w:
        q_ref, s_ref = oracle_weight(w_cpu, per_channel, fmt=fmt_w)
        assert_scale_equal(s_w, s_ref, f"s_w {fmt_w}")
        assert_codes_equal(qw, q_ref, K, f"qW {fmt_w}")
    return y


@pytest.mark.parametrize("fmt_a,fmt_w", PAIRS)
@pytest.mark.parametrize("M", [1, 9, 16, 40, 300])
def test_linear_formats(fmt_a, fmt_w, M):
    K, N = 1000, 1027
    a = I.activations_normal(M, K, (179, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (180,))
    b = I.bias_normal(N, (181,))
    path = "gemv" if F.fp8_uses_gemv(M, K, N) else "gemm"
    for per_channel in (False, True):
        y = run_ex(a, w, fmt_a, fmt_w, per_channel, b)
        linear_parity(y, a, w, per_channel, b, what=f"{path} M={M} {fmt_a}x{fmt_w} pc={per_channel}",
                      fmt_a=fmt_a, fmt_w=fmt_w)


@pytest.mark.parametrize("fmt_a,fmt_w", PAIRS)
def test_linear_formats_large_k(fmt_a, fmt_w):
    """down_proj-shaped K (14336: 8-rank GEMV clusters) and a multi-tile GEMM."""
    for M, N in ((8, 1100), (700, 600)):
        K = 14336
        a = I.activations_heavy_tail(M, K, (182, M))
        w = I.weights_row_std(N, K, (183, N))
        y = run_ex(a, w, fmt_a, fmt_w, True)
        linear_parity(y, a, w, True, what=f"K=14336 M={M} {fmt_a}x{fmt_w}", fmt_a=fmt_a, fmt_w=fmt_w)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [3, 16, 200])
@pytest.mark.parametrize("factor", [0.2, 1.5])
def test_linear_static_scale(fmt, M, factor):
    K, N = 2050, 3001
    a = I.activations_normal(M, K, (184, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (185,))
    s = np.float32(float(O.amax(f32(a))) / O.fp8_max(fmt) * factor)
    y = run_ex(a, w, fmt, fmt, False, None, s_static=s)
    linear_parity(y, a, w, False, what=f"static {fmt} M={M} x{factor}", fmt_a=fmt, fmt_w=fmt, s_static=s)


@pytest.mark.parametrize("M", [4, 256])
def test_static_with_dynamic_value_matches_dynamic_bit_for_bit(M):
    """Given the scale the dynamic path derives, the static path computes the same codes with
    the same kernels: Y must be identical, through fp8_linear_static as well."""
    K, N = 1024, 777
    a = I.activations_normal(M, K, (186, M)).to(DEV)
    qw, s_w = F.fp8_quantize_weight(I.weights_normal(N, K, (187,)).to(DEV))
    _, s_dyn = F.fp8_quantize_act(a)
    y_dyn = F.fp8_linear(a, qw, s_w)
    y_st = F.fp8_linear_static(a, s_dyn, qw, s_w)
    y_ex = F.fp8_linear_ex(a, qw, s_w, s_static=s_dyn)
    torch.cuda.synchronize()
    assert torch.equal(y_dyn, y_st) and torch.equal(y_dyn, y_ex)


@pytest.mark.parametrize("fmt_a,fmt_w", PAIRS)
def test_scaled_mm_formats_equal_linear(fmt_a, fmt_w):
    for M in (5, 130):
        K, N = 512, 640
        a = I.activations_normal(M, K, (188, M)).to(DEV)
        qw, s_w = F.fp8_quantize_weight_ex(I.weights_normal(N, K, (189,)).to(DEV), fmt_w)
        qa, s_a = F.fp8_quantize_act_ex(a, fmt_a)
        y1 = F.fp8_scaled_mm_ex(qa, fmt_a, K, s_a, qw, fmt_w, s_w)
        # the least workspace: no K split, the GEMM sums in fp8_scaled_mm's order
        ws = torch.empty(max(1, F.min_workspace_bytes(M, K, N)), dtype=torch.uint8, device=DEV)
        y2 = F.fp8_linear_ex(a, qw, s_w, fmt_a=fmt_a, fmt_w=fmt_w, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), (M, fmt_a, fmt_w)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("M,K", [(1, 4096), (16, 14336)])
def test_gemv_in_kernel_codes_identity_weights(fmt, static, M, K):
    """W = I: Y[m, n] = bf16(s_a * s_w * dec(qA[m, n])) is one product, so every code the GEMV
    chose inside the kernel is visible in Y (neighbouring codes differ by >= 12.5%)."""
    g = np.random.default_rng(190 + M)
    a = (g.standard_normal((M, K)) * np.exp2(g.integers(-14, 9, (M, K)))).astype(np.float32)
    a = I.to_bf16(a)
    w = torch.eye(K, dtype=torch.bfloat16)
    s = np.float32(float(O.amax(f32(a))) / O.fp8_max(fmt) / 2) if static else None
    y = run_ex(a, w, fmt, "e4m3", False, None, s_static=s, check_w=False)
    cols = np.sort(g.choice(K, 600, replace=False))
    linear_parity(y, a, w, False, cols=cols, what=f"identity {fmt} static={static}", fmt_a=fmt, fmt_w="e4m3",
                  s_static=s)


def test_invalid_format_rejected():
    a = torch.zeros((2, 32), dtype=torch.bfloat16, device=DEV)
    qw, s_w = F.fp8_quantize_weight(torch.zeros((8, 32), dtype=torch.bfloat16, device=DEV))
    y = torch.empty((2, 8), dtype=torch.bfloat16, device=DEV)
    st = F.lib().fp8_linear_ex(a.data_ptr(), 2, 32, 32, 2, None, qw.data_ptr(), 0, 8, qw.stride(0), s_w.data_ptr(),
                               0, None, y.data_ptr(), 8, None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == F.FP8_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [1, 7, 16])
def test_gemv_quantizer_on_rounding_boundaries(fmt, M):
    """Activations made of FP8 rounding midpoints with amax = max(fmt), so s_a = 1 and every
    quotient lies exactly on a boundary: the in-kernel quantizer's fast path must refuse every
    unit and the exact division (queued, and inline once the queue is full) must decide.
    Identity weights make every chosen code visible in Y."""
    K = 4096
    g = np.random.default_rng(400 + M)
    table = O.E4M3_DECODE[:0x7F] if fmt == "e4m3" else O.E5M2_DECODE[:0x7C]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    mids = mids[np.abs(mids) < O.fp8_max(fmt)]
    a = g.choice(mids, size=(M, K)) * np.where(g.random((M, K)) < 0.5, -1, 1).astype(np.float32)
    a[0, 0] = O.fp8_max(fmt)
    a = I.to_bf16(a.astype(np.float32))
    assert float(O.amax(f32(a))) == O.fp8_max(fmt)
    w = torch.eye(K, dtype=torch.bfloat16)
    y = run_ex(a, w, fmt, "e4m3", False, None, check_w=False)
    cols = np.sort(g.choice(K, 512, replace=False))
    linear_parity(y, a, w, False, cols=cols, what=f"boundaries {fmt} M={M}", fmt_a=fmt, fmt_w="e4m3")
