"""GPU parity of the quantization kernels: e4m3 codes and fp32 scales must be bit-exact."""

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from parity import assert_codes_equal, assert_scale_equal, oracle_act, oracle_weight

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    F.lib()


def all_finite_bf16() -> torch.Tensor:
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return bits[torch.isfinite(bits.float())]


def run_act(a_cpu: torch.Tensor, lda_pad: int = 0):
    M, K = a_cpu.shape
    if lda_pad:
        big = torch.zeros((M, K + lda_pad), dtype=torch.bfloat16)
        big[:, :K] = a_cpu
        a = big.to(DEV)[:, :K]
    else:
        a = a_cpu.to(DEV)
    qa, s_a = F.fp8_quantize_act(a)
    torch.cuda.synchronize()
    return qa, s_a


def check_act(a_cpu, what, lda_pad=0):
    qa, s_a = run_act(a_cpu, lda_pad)
    q_ref, s_ref = oracle_act(a_cpu)
    assert_scale_equal(s_a, s_ref, what)
    assert_codes_equal(qa, q_ref, a_cpu.shape[1], what)


def test_every_bf16_value_with_unit_scale():
    x = all_finite_bf16()
    x = x[x.float().abs() <= 448]
    x = torch.cat([x, torch.tensor([448.0], dtype=torch.bfloat16)])
    pad = (-x.numel()) % 256
    a = torch.cat([x, torch.zeros(pad, dtype=torch.bfloat16)]).view(-1, 256)
    qa, s_a = run_act(a)
    assert s_a.item() == 1.0
    check_act(a, "all bf16 in [-448, 448], s = 1")


def test_every_bf16_value_with_huge_scale():
    x = all_finite_bf16()
    pad = (-x.numel()) % 255
    a = torch.cat([x, torch.zeros(pad, dtype=torch.bfloat16)]).view(-1, 255)  # K not a multiple of 16
    check_act(a, "all finite bf16")


@pytest.mark.parametrize("mag", [1e-38, 3e-36, 1e-3, 1.0, 7e4, 1e30])
def test_scales_across_magnitudes(mag):
    g = np.random.default_rng(int(np.log10(mag) + 100))
    a = I.to_bf16(g.standard_normal((37, 1000)).astype(np.float32) * np.float32(mag))
    check_act(a, f"magnitude {mag}")


def test_tiny_config_activations():
    c = I.tiny_case()
    check_act(c.a, c.name)


@pytest.mark.parametrize("idx", range(4))
def test_unaligned_config_activations(idx):
    c = I.unaligned_cases()[idx]
    check_act(c.a, c.name)
    check_act(c.a, c.name + " strided", lda_pad=3)


def test_prefill_sized_activations():
    a = I.prefill_activations(3, M=2048)  # down_proj K = 14336, heavy-tailed channels
    check_act(a, "prefill down 2048x14336")


@pytest.mark.parametrize("M,K,pad", [(64, 4096, 0), (65, 4096, 0), (64, 4096, 5), (1, 262144, 0), (17, 15421, 0),
                                     (40, 1000, 3)])
def test_activation_quantization_shapes(M, K, pad):
    """Gap-free and strided rows, one long row, ragged K, grids from a few CTAs to hundreds:
    bit-exact codes and scale."""
    a = I.activations_heavy_tail(M, K, (960, M, K))
    check_act(a, f"{M}x{K} pad={pad}", lda_pad=pad)


def test_zero_activations():
    qa, s_a = run_act(torch.zeros((5, 33), dtype=torch.bfloat16))
    assert s_a.item() == 1.0 and not qa.any()


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("shape", [(256, 256), (4097, 4100), (3001, 2050), (1027, 1000), (4096, 4096)])
def test_weight_quantization(per_channel, shape):
    N, K = shape
    w = I.weights_row_std(N, K, (77, N, K))
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=per_channel)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_weight(w, per_channel)
    what = f"W {shape} per_channel={per_channel}"
    assert_scale_equal(s_w, s_ref, what)
    assert_codes_equal(qw, q_ref, K, what)


def test_weight_rows_with_zero_and_tiny_rows():
    w = I.weights_normal(64, 200, (78,)).float()
    w[3] = 0
    w[5] *= 1e-36
    w = w.bfloat16()
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=True)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_weight(w, True)
    assert_scale_equal(s_w, s_ref, "zero/tiny rows")
    assert_codes_equal(qw, q_ref, 200, "zero/tiny rows")
    assert s_w[3].item() == 1.0


def test_quantization_is_deterministic():
    a = I.prefill_activations(0, M=512).to(DEV)
    q1, s1 = F.fp8_quantize_act(a)
    q2, s2 = F.fp8_quantize_act(a)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_all_bf16_values_under_many_scales():
    """Every finite bf16 value at 40 scales (random amax and powers of two, whose quotients
    land exactly on e4m3 rounding midpoints): codes and scale bit-exact."""
    x = all_finite_bf16()
    g = np.random.default_rng(21)
    targets = [float(v) for v in g.standard_normal(28) * np.exp2(g.integers(-40, 40, 28))]
    targets += [448.0 * 2.0 ** k for k in (-20, -9, -6, -3, -1, 0, 1, 2, 5, 9, 17, 30)]
    for T in targets:
        T = abs(float(torch.tensor(T).bfloat16().float()))
        v = x[x.float().abs() <= T]
        v = torch.cat([v, torch.tensor([T, -T], dtype=torch.bfloat16)])
        pad = (-v.numel()) % 240
        a = torch.cat([v, torch.zeros(pad, dtype=torch.bfloat16)]).view(-1, 240)
        check_act(a, f"all bf16 with amax {T:g}")
