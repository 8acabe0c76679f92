"""C-ABI boundary tests that need no GPU.

The library is built here (nvcc cross-compiles for sm_103a) and loaded with ctypes.
Only host logic runs: symbol exports, size/layout helpers, status strings, and argument
validation, which must reject bad input synchronously before any CUDA call.
"""

import os
import re

import pytest

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return F.lib()


def declared_functions():
    names = set()
    for h in os.listdir(INCLUDE):
        if not h.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fp8_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("fp8_quantize_weight", "fp8_quantize_act", "fp8_linear", "fp8_linear_channelwise",
                     "fp8_scaled_mm", "fp8_workspace_bytes", "fp8_last_device_status", "fp8_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_binding_names_match_c_abi():
    for name in declared_functions():
        assert callable(getattr(F, name)), name


def test_status_strings(L):
    for code, name in [(0, "FP8_OK"), (1, "FP8_ERR_INVALID_ARG"), (2, "FP8_ERR_MISALIGNED"),
                       (3, "FP8_ERR_WORKSPACE"), (4, "FP8_ERR_CUDA"), (5, "FP8_ERR_TIMEOUT"),
                       (6, "FP8_ERR_UNSUPPORTED_DEVICE")]:
        assert F.status_string(code) == name
    assert F.status_string(99) == "FP8_ERR_UNKNOWN"


@pytest.mark.parametrize("K", [0, 1, 15, 16, 17, 1000, 4095, 4096, 4100, 14336])
def test_min_ld(L, K):
    assert F.fp8_min_ld(K) == F.min_ld(K)
    assert F.fp8_min_ld(K) % 16 == 0 and F.fp8_min_ld(K) >= max(K, 16)


def test_workspace_and_dispatch(L):
    base = F.FP8_QUANT_WORKSPACE_BYTES
    # decode shapes run the GEMV, which quantizes A itself: no workspace
    for M in (1, 2, 8, 15, 16):
        assert F.fp8_uses_gemv(M, 4096, 4096)
        assert F.fp8_workspace_bytes(M, 4096, 4096) == 0
    # GEMM shapes hold the partial amax values, s_a and qA [M, min_ld(K)]; small M adds the
    # split-K fp32 partials [splits, M, N rounded up to 4] from the next 256-byte boundary
    for M, K in ((33, 8192), (16384, 14336), (100, 4100)):
        assert not F.fp8_uses_gemv(M, K, 4096)
        assert F.min_workspace_bytes(M, K, 4096) == base + M * F.min_ld(K)
        ws = F.fp8_workspace_bytes(M, K, 4096)
        assert ws >= base + M * F.min_ld(K)
        if ws > base + M * F.min_ld(K):
            split = ws - (base + M * F.min_ld(K) + 255) // 256 * 256
            assert split > 0 and split % (M * 4096 * 4) == 0 and 2 <= split // (M * 4096 * 4) <= 16
    assert F.fp8_workspace_bytes(16384, 14336, 4096) == base + 16384 * F.min_ld(14336)  # enough tiles: no split
    assert F.fp8_workspace_bytes(33, 8192, 4096) > F.min_workspace_bytes(33, 8192, 4096)  # one row block: split
    assert F.fp8_workspace_bytes(0, 4096, 4096) == 0
    assert not F.fp8_uses_gemv(4, 40000, 4096)  # K beyond the GEMV's slice budget -> GEMM


# ---------------------------------------------------------------------------
# argument validation (fake, never dereferenced device addresses)
# ---------------------------------------------------------------------------

P = 0x7F0000000000  # 256-byte aligned fake address
WS = 0x7F0000100000


def lin(L, a=P, M=4, K=64, lda=64, qw=P, N=32, ldqw=64, s_w=P, bias=None, y=P, ldy=32, ws=WS,
        ws_bytes=1 << 20, channelwise=False):
    fn = L.fp8_linear_channelwise if channelwise else L.fp8_linear
    return fn(a, M, K, lda, qw, N, ldqw, s_w, bias, y, ldy, ws, ws_bytes, None)


@pytest.mark.parametrize("channelwise", [False, True])
def test_linear_rejects_bad_arguments(L, channelwise):
    c = dict(channelwise=channelwise)
    assert lin(L, a=None, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, qw=None, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, y=None, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, s_w=None, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, M=-1, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, K=-1, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, N=-5, **c) == F.FP8_ERR_INVALID_ARG
    assert lin(L, lda=63, **c) == F.FP8_ERR_INVALID_ARG           # lda < K
    assert lin(L, ldy=31, **c) == F.FP8_ERR_INVALID_ARG           # ldy < N
    assert lin(L, ldqw=48, **c) == F.FP8_ERR_INVALID_ARG          # ldqw < K
    assert lin(L, K=60, lda=60, ldqw=72, **c) == F.FP8_ERR_MISALIGNED  # FP8 ld not a multiple of 16
    assert lin(L, qw=P + 8, **c) == F.FP8_ERR_MISALIGNED          # FP8 base not 16-byte aligned
    assert lin(L, a=P + 1, **c) == F.FP8_ERR_MISALIGNED           # bf16 base odd
    assert lin(L, bias=P + 1, **c) == F.FP8_ERR_MISALIGNED
    # GEMM-path shapes (M > 16) need a workspace with room for qA
    assert lin(L, M=64, ws=None, **c) == F.FP8_ERR_WORKSPACE
    assert lin(L, M=64, ws_bytes=100, **c) == F.FP8_ERR_WORKSPACE
    assert lin(L, M=64, ws=WS + 16, **c) == F.FP8_ERR_WORKSPACE   # not 256-byte aligned
    need = F.fp8_workspace_bytes(64, 64, 32)
    assert lin(L, M=64, ws_bytes=need - 1, **c) == F.FP8_ERR_WORKSPACE


def test_linear_empty_is_noop_without_device(L):
    # M == 0 or N == 0 returns before any CUDA call (no GPU in this container)
    assert lin(L, M=0, a=None, y=None) == F.FP8_OK
    assert lin(L, N=0, qw=None, ldy=1, s_w=None) == F.FP8_OK


def test_quantize_calls_reject_bad_arguments(L):
    q = L.fp8_quantize_weight
    assert q(None, 8, 64, 64, 0, P, 64, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG
    assert q(P, 8, 64, 64, 2, P, 64, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG   # bad flag
    assert q(P, 8, 64, 64, 0, P, 64, None, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG
    assert q(P, 8, 64, 64, 0, P, 64, P, WS, 16, None) == F.FP8_ERR_WORKSPACE
    assert q(P, 8, 64, 64, 0, P, 40, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG   # ldq < K
    assert q(P, 8, 64, 64, 1, P, 64, P, None, 0, None) != F.FP8_ERR_WORKSPACE       # per-channel: no ws
    a = L.fp8_quantize_act
    assert a(P, 8, 64, 32, P, 64, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG      # lda < K
    assert a(P, 8, 64, 64, P + 4, 64, P, WS, 1 << 16, None) == F.FP8_ERR_MISALIGNED
    assert a(P, 8, 64, 64, P, 64, None, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG
    s = L.fp8_scaled_mm
    assert s(P, 4, 64, 64, None, P, 8, 64, P, 0, None, P, 8, None) == F.FP8_ERR_INVALID_ARG
    assert s(P, 4, 64, 64, P, P, 8, 64, P, 3, None, P, 8, None) == F.FP8_ERR_INVALID_ARG
    assert s(P, 4, 64, 24, P, P, 8, 64, P, 0, None, P, 8, None) == F.FP8_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(L):
    # validation passes, then the device query fails: no crash, an error code
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lin(L) in (F.FP8_ERR_CUDA, F.FP8_ERR_UNSUPPORTED_DEVICE)


def test_wider_calls_reject_bad_formats_and_scales(L):
    """Format values other than FP8_E4M3 / FP8_E5M2 and a missing static scale are refused
    before anything touches a device."""
    ex = L.fp8_linear_ex
    args = lambda fa, fw, s=None, pc=0: (P, 4, 64, 64, fa, s, P, fw, 32, 64, P, pc, None, P, 32, WS, 1 << 20, None)
    for fa, fw in ((2, 0), (0, 2), (-1, 1), (1, 7)):
        assert ex(*args(fa, fw)) == F.FP8_ERR_INVALID_ARG
    assert ex(*args(0, 0, pc=2)) == F.FP8_ERR_INVALID_ARG
    assert ex(*args(0, 0, s=P + 2)) == F.FP8_ERR_MISALIGNED      # static scale not 4-byte aligned
    st = L.fp8_linear_static
    assert st(P, 4, 64, 64, None, P, 32, 64, P, 0, None, P, 32, WS, 1 << 20, None) == F.FP8_ERR_INVALID_ARG
    qw = L.fp8_quantize_weight_ex
    assert qw(P, 8, 64, 64, 0, 3, P, 64, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG
    qa = L.fp8_quantize_act_ex
    assert qa(P, 8, 64, 64, 5, None, P, 64, P, WS, 1 << 16, None) == F.FP8_ERR_INVALID_ARG
    assert qa(P, 8, 64, 64, 1, None, P, 64, P, WS, 16, None) == F.FP8_ERR_WORKSPACE   # dynamic needs ws
    assert qa(P, 8, 64, 64, 1, P + 1, P, 64, P, None, 0, None) == F.FP8_ERR_MISALIGNED
    sm = L.fp8_scaled_mm_ex
    assert sm(P, 9, 4, 64, 64, P, P, 0, 8, 64, P, 0, None, P, 8, None) == F.FP8_ERR_INVALID_ARG
    assert sm(P, 0, 4, 64, 64, P, P, 9, 8, 64, P, 0, None, P, 8, None) == F.FP8_ERR_INVALID_ARG


def test_static_quantize_needs_no_workspace(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # static scale: validation passes without a workspace; only the device query fails here
    assert L.fp8_quantize_act_ex(P, 8, 64, 64, 0, P, P, 64, P, None, 0, None) in (
        F.FP8_ERR_CUDA, F.FP8_ERR_UNSUPPORTED_DEVICE)


def test_selftest_rejects_bad_limits(L):
    for limit in (-1, 0, 999, 10_000_000_001):
        assert L.fp8_selftest_timeout(limit, None) == F.FP8_ERR_INVALID_ARG


def wo(L, a=P, M=4, K=64, lda=64, qw=P, fmt_w=0, N=32, ldqw=64, s_w=P, per_channel=0, bias=None, y=P, ldy=32,
       ws=WS, ws_bytes=1 << 20):
    return L.fp8_linear_weight_only(a, M, K, lda, qw, fmt_w, N, ldqw, s_w, per_channel, bias, y, ldy, ws, ws_bytes,
                                    None)


def test_weight_only_rejects_bad_arguments(L):
    """fp8_linear_weight_only validates before any device work: formats, flags, pointers,
    strides, alignment, and the workspace its GEMM path needs; empty shapes are no-ops."""
    assert wo(L, fmt_w=2) == F.FP8_ERR_INVALID_ARG
    assert wo(L, fmt_w=-1) == F.FP8_ERR_INVALID_ARG
    assert wo(L, per_channel=2) == F.FP8_ERR_INVALID_ARG
    assert wo(L, a=None) == F.FP8_ERR_INVALID_ARG
    assert wo(L, qw=None) == F.FP8_ERR_INVALID_ARG
    assert wo(L, y=None) == F.FP8_ERR_INVALID_ARG
    assert wo(L, s_w=None) == F.FP8_ERR_INVALID_ARG
    assert wo(L, lda=63) == F.FP8_ERR_INVALID_ARG                # lda < K
    assert wo(L, ldy=31) == F.FP8_ERR_INVALID_ARG                # ldy < N
    assert wo(L, ldqw=48) == F.FP8_ERR_INVALID_ARG               # ldqw < K
    assert wo(L, K=60, lda=60, ldqw=72) == F.FP8_ERR_MISALIGNED  # FP8 ld not a multiple of 16
    assert wo(L, qw=P + 8) == F.FP8_ERR_MISALIGNED
    assert wo(L, a=P + 1) == F.FP8_ERR_MISALIGNED
    assert wo(L, bias=P + 1) == F.FP8_ERR_MISALIGNED
    # GEMM-path shapes hold the up-converted weights in the workspace
    need = F.fp8_weight_only_workspace_bytes(64, 64, 32)
    assert need > 0
    assert wo(L, M=64, ws=None, ws_bytes=0) == F.FP8_ERR_WORKSPACE
    assert wo(L, M=64, ws_bytes=need - 1) == F.FP8_ERR_WORKSPACE
    assert wo(L, M=64, ws=WS + 16) == F.FP8_ERR_WORKSPACE        # not 256-byte aligned
    # decode shapes need none, and empty shapes return before any CUDA call
    assert F.fp8_weight_only_workspace_bytes(4, 4096, 4096) == 0
    assert wo(L, M=0, a=None, y=None) == F.FP8_OK
    assert wo(L, N=0, qw=None, s_w=None, ldy=1) == F.FP8_OK


def test_crossover_rule(L):
    """M <= 32 runs the GEMV by default (the crossover): up to 16 tokens it quantizes A itself
    (no workspace), from 17 on A is quantized once into the workspace first (no split-K
    partials). fp8_set_gemv_max_m moves the crossover (32 at most; 0 sends everything to the
    GEMM), and K beyond 32768 always takes the GEMM."""
    import os
    prev = F.fp8_set_gemv_max_m(-1)
    if "FP8W8A8_GEMV_MAX_M" not in os.environ:
        assert prev == 32
    try:
        F.fp8_set_gemv_max_m(32)
        assert F.fp8_uses_gemv(32, 14336, 28672) and not F.fp8_uses_gemv(33, 2048, 2560)
        assert not F.fp8_uses_gemv(1, 40000, 2048)
        base = F.FP8_QUANT_WORKSPACE_BYTES
        assert F.fp8_workspace_bytes(16, 2048, 2560) == 0
        assert F.fp8_workspace_bytes(32, 2048, 2560) == F.min_workspace_bytes(32, 2048, 2560) == base + 32 * 2048
        assert F.fp8_workspace_bytes(33, 8192, 4096) > F.min_workspace_bytes(33, 8192, 4096)  # GEMM: partials
        F.fp8_set_gemv_max_m(16)
        assert F.fp8_uses_gemv(16, 4096, 4096) and not F.fp8_uses_gemv(17, 2048, 2560)
        F.fp8_set_gemv_max_m(8)
        assert not F.fp8_uses_gemv(9, 2048, 2560)
        F.fp8_set_gemv_max_m(0)
        assert not F.fp8_uses_gemv(1, 2048, 2560)
    finally:
        F.fp8_set_gemv_max_m(prev)
