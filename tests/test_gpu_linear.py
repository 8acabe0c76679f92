"""GPU parity of the W8A8 linear (decode GEMV and tcgen05 GEMM paths) against the oracle.

Y must lie within one bf16 ulp of the exact value plus K * 2^-23 * sum_k |a_k w_k|
(oracle.tolerance); the GPU's qW / s_w are checked bit-exact where the test quantizes
them. Output buffers carry canary guard bands to catch stray writes.
"""

import functools

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import _build
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I
from parity import (assert_codes_equal, assert_guards_intact, assert_scale_equal, guarded, linear_parity,
                    oracle_weight, tail_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    F.lib()


def run_linear(a_cpu, w_cpu, per_channel, bias_cpu=None, guard=True, lda_pad=0):
    """Quantize W on the GPU, run the linear (into a guarded Y buffer), return (y, qw, s_w)."""
    M, K = a_cpu.shape
    N = w_cpu.shape[0]
    qw, s_w = F.fp8_quantize_weight(w_cpu.to(DEV), per_channel=per_channel)
    if lda_pad:
        big = torch.zeros((M, K + lda_pad), dtype=torch.bfloat16)
        big[:, :K] = a_cpu
        a = big.to(DEV)[:, :K]
    else:
        a = a_cpu.to(DEV)
    bias = None if bias_cpu is None else bias_cpu.to(DEV)
    fn = F.fp8_linear_channelwise if per_channel else F.fp8_linear
    if guard:
        buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
        fn(a, qw, s_w, bias, out=y)
        torch.cuda.synchronize()
        assert_guards_intact(buf, base, row_bytes, used, M)
    else:
        y = fn(a, qw, s_w, bias)
        torch.cuda.synchronize()
    assert F.fp8_last_device_status() == F.FP8_OK
    return y, qw, s_w


def check(a, w, per_channel, bias=None, what="", rows=None, cols=None, lda_pad=0, check_w=True):
    y, qw, s_w = run_linear(a, w, per_channel, bias, lda_pad=lda_pad)
    if check_w:
        q_ref, s_ref = oracle_weight(w, per_channel, None if cols is None else np.asarray(cols))
        sel = slice(None) if cols is None else torch.as_tensor(np.asarray(cols), device=DEV)
        assert_scale_equal(s_w if not per_channel else s_w[sel], s_ref, what + " s_w")
        assert_codes_equal(qw[sel], q_ref, w.shape[1], what + " qW")
    return linear_parity(y, a, w, per_channel, bias, rows, cols, what)


# --------------------------------------------------------------------------- decode GEMV

@pytest.mark.parametrize("M", list(range(1, 17)))
def test_gemv_every_m(M):
    K, N = 1000, 1027
    assert F.fp8_uses_gemv(M, K, N)
    a = I.activations_normal(M, K, (901, M), outlier_cols=4)
    w = I.weights_row_std(N, K, (902,))
    b = I.bias_normal(N, (903,))
    check(a, w, False, b, f"gemv M={M} per-tensor")
    check(a, w, True, None, f"gemv M={M} channelwise", check_w=False)


def test_tiny_config():
    c = I.tiny_case()
    check(c.a, c.w, c.per_channel, None, c.name)


@pytest.mark.parametrize("idx", range(4))
def test_unaligned_config(idx):
    c = I.unaligned_cases()[idx]
    check(c.a, c.w, c.per_channel, None, c.name)
    check(c.a, c.w, True, I.bias_normal(c.N, (904,)), c.name + " channelwise+bias", lda_pad=5, check_w=False)


@pytest.mark.parametrize("layer", range(4))
@pytest.mark.parametrize("M", list(I.DECODE_MS))
def test_decode_config_layers(layer, M):
    """Mistral-7B decode layers at full size; Y checked on all rows and 1536 sampled columns."""
    L = I.LLAMA8B_LAYERS[layer]
    w = I.decode_weight(layer)
    a = I.decode_activations(M, layer)
    cols = np.unique(np.concatenate([np.random.default_rng(layer).choice(L.N, 1536, replace=False),
                                     [0, L.N - 1]]))
    check(a, w, False, None, f"decode {L.name} M={M}", cols=cols)


# --------------------------------------------------------------------------- prefill GEMM

@pytest.mark.parametrize("M,K,N", [(40, 4096, 6401), (33, 256, 256), (128, 128, 256), (130, 1000, 1027), (300, 4100, 257),
                                   (257, 2050, 3001), (512, 4096, 512), (1000, 96, 520)])
@pytest.mark.parametrize("per_channel", [False, True])
def test_gemm_ragged(M, K, N, per_channel):
    assert not F.fp8_uses_gemv(M, K, N)
    a = I.activations_heavy_tail(M, K, (905, M, K))
    w = I.weights_row_std(N, K, (906, N, K))
    b = I.bias_normal(N, (907, N))
    check(a, w, per_channel, b, f"gemm {M}x{K}x{N} pc={per_channel}")


def _tail_case(split, K=520, N=2500):
    """One GEMM whose last wave is split by columns into `split` units per tile (the process's
    FP8W8A8_GEMM_TAIL allows it), parity-checked against the oracle; the mode (pairs or one CTA
    per tile) is whatever the process's switches give."""
    qa0 = torch.zeros((4096, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    qw0 = torch.zeros((N, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    cfg0 = F.fp8_gemm_config(qa0, qw0, K)
    two = cfg0["two_sm"]
    slots = cfg0["grid"] // (2 if two else 1)
    assert slots <= torch.cuda.get_device_properties(0).multi_processor_count
    M = tail_rows((N + 255) // 256, slots, split, 256 if two else 128)
    cfg = F.fp8_gemm_config(qa0[:M], qw0, K, F.fp8_workspace_bytes(M, K, N))  # the workspace fp8_linear takes
    assert cfg["tail_split"] == split and cfg["splits"] == 1, cfg
    a = I.activations_heavy_tail(M, K, (931, M, split))
    w = I.weights_row_std(N, K, (932, N))
    b = I.bias_normal(N, (933, N))
    check(a, w, True, b, f"tail split {split} {M}x{K}x{N} two_sm={two}", check_w=False)


def _in_child(call, **env):
    """Runs `call` (an expression over this module, as t) in a fresh process with extra
    environment switches (read once per process by the library)."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = f"import sys; sys.path[:0] = [{here!r}, {os.path.dirname(here)!r}]\nimport test_gpu_linear as t\n{call}\n"
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


def test_gemm_tail_split_pairs():
    """CTA pairs: the last, partial wave's tiles divided by columns into 2 units over all of K
    (ragged M, N and K, per-channel scales, bias), against the oracle with guard bands."""
    _tail_case(2)


@pytest.mark.parametrize("pair,split", [("1", 4), ("0", 2), ("0", 4)])
def test_gemm_tail_split_other_modes(pair, split):
    """The same with quarters (FP8W8A8_GEMM_TAIL=4) and with one CTA per tile
    (FP8W8A8_GEMM_PAIR=0), each in a child process."""
    _in_child(f"t._tail_case({split})", FP8W8A8_GEMM_PAIR=pair, FP8W8A8_GEMM_TAIL=str(split))


@pytest.mark.parametrize("M,K,N,f", [(100, 2048, 2560, 4), (300, 1000, 1027, 4), (257, 2050, 3001, 2)])
def test_gemm_fill_split(M, K, N, f):
    """Few tiles and short K: every tile of the one partial wave split by columns into f units
    over all of K (one CTA per tile, and CTA pairs with a ragged second row block; four units
    while they fit one wave of the 76 pairs / 152 CTAs, else two), per-channel scales and bias,
    against the oracle with guard bands."""
    qa = torch.zeros((M, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    qw = torch.zeros((N, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    cfg = F.fp8_gemm_config(qa, qw, K, F.fp8_workspace_bytes(M, K, N))
    assert cfg["splits"] == 1 and cfg["tail_split"] == f, cfg
    a = I.activations_heavy_tail(M, K, (934, M))
    w = I.weights_row_std(N, K, (935, N))
    b = I.bias_normal(N, (936, N))
    check(a, w, True, b, f"fill split {M}x{K}x{N}", check_w=False)


def test_gemm_strided_activations_and_output():
    M, K, N = 200, 1000, 300
    a = I.activations_normal(M, K, (908,))
    w = I.weights_normal(N, K, (909,))
    check(a, w, True, None, "gemm strided A", lda_pad=24, check_w=False)
    # odd ldy: scalar epilogue stores
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=True)
    ybig = torch.full((M, N + 3), 7.0, dtype=torch.bfloat16, device=DEV)
    F.fp8_linear_channelwise(a.to(DEV), qw, s_w, out=ybig[:, :N])
    torch.cuda.synchronize()
    assert torch.all(ybig[:, N:] == 7.0)
    linear_parity(ybig[:, :N], a, w, True, what="gemm odd ldy")


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_prefill_config_full_size_sampled(layer):
    """Llama-3-8B prefill layer at M = 16384, channelwise, as the benchmark runs it.
    qW/s_w bit-exact on sampled rows; Y on 40 sampled rows x 768 sampled columns."""
    L = I.LLAMA8B_LAYERS[layer]
    w = I.prefill_weight(layer)
    a = I.prefill_activations(layer)
    g = np.random.default_rng(100 + layer)
    rows = np.unique(np.concatenate([g.choice(a.shape[0], 38, replace=False), [0, a.shape[0] - 1]]))
    cols = np.unique(np.concatenate([g.choice(L.N, 766, replace=False), [0, L.N - 1]]))
    y, qw, s_w = run_linear(a, w, True, guard=False)
    q_ref, s_ref = oracle_weight(w, True, cols)
    sel = torch.as_tensor(cols, device=DEV)
    assert_scale_equal(s_w[sel], s_ref, "prefill s_w")
    assert_codes_equal(qw[sel], q_ref, L.K, "prefill qW")
    linear_parity(y, a, w, True, None, rows, cols, f"prefill {L.name}")


@functools.lru_cache(maxsize=None)
def _tinyllama_layer(depth, li, per_channel):
    """Host weights of one TinyLlama linear, their oracle quantization on sampled columns, and
    the library's quantized copy on the device (shared by every M of the sweep)."""
    L = I.TINYLLAMA_LAYERS[li]
    w = I.tinyllama_weight(depth, li)
    cols = np.unique(np.r_[np.random.default_rng(7 + li).choice(L.N, 384, replace=False), 0, L.N - 1])
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=per_channel)
    return w, cols, oracle_weight(w, per_channel, cols), qw, s_w


@pytest.mark.parametrize("depth", [0, I.TINYLLAMA_DEPTH - 1])
@pytest.mark.parametrize("M", sorted(set(I.TINYLLAMA_MS) | {17, 33}))
def test_tinyllama_sweep_sampled(M, depth):
    """Every M of the TinyLlama sweep, plus M = 17 (the first row count the GEMV runs on
    activations quantized beforehand) and 33 (the first on the GEMM), first and last layer of
    the stack, both weight modes: Y against the oracle on sampled rows (all rows up to M = 64)
    and 386 sampled columns."""
    from parity import assert_y_within_tolerance, f32, oracle_act
    for li, L in enumerate(I.TINYLLAMA_LAYERS):
        a = I.tinyllama_activations(M, depth, li)
        rows = np.arange(M) if M <= 64 else np.unique(np.r_[np.random.default_rng(M).choice(M, 30), M - 1])
        qa, s_a = oracle_act(a, rows)
        ad = a.to(DEV)
        for pc in (False, True):
            w, cols, (qw_o, s_w_o), qw, s_w = _tinyllama_layer(depth, li, pc)
            fn = F.fp8_linear_channelwise if pc else F.fp8_linear
            y = fn(ad, qw, s_w)
            torch.cuda.synchronize()
            assert F.fp8_last_device_status() == F.FP8_OK
            assert_y_within_tolerance(f32(y)[np.ix_(rows, cols)], qa, s_a, qw_o, s_w_o, None,
                                      f"tinyllama d={depth} {L.name} M={M} pc={pc}")


# --------------------------------------------------------------------------- API behaviour

@pytest.mark.parametrize("M", [4, 300])
def test_scaled_mm_equals_linear(M):
    K, N = 2050, 777
    a = I.activations_normal(M, K, (910, M)).to(DEV)
    w = I.weights_row_std(N, K, (911,)).to(DEV)
    qw, s_w = F.fp8_quantize_weight(w, per_channel=True)
    # the least workspace: no K split, so the GEMM sums in the same order as fp8_scaled_mm
    ws = torch.empty(max(1, F.min_workspace_bytes(M, K, N)), dtype=torch.uint8, device=DEV)
    y1 = F.fp8_linear_channelwise(a, qw, s_w, ws=ws)
    qa, s_a = F.fp8_quantize_act(a)
    y2 = F.fp8_scaled_mm(qa, K, s_a, qw, s_w, per_channel=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M", [3, 200])
def test_k_zero_gives_bias(M):
    N = 300
    a = torch.empty((M, 0), dtype=torch.bfloat16, device=DEV)
    qw = torch.zeros((N, 16), dtype=torch.uint8, device=DEV)
    s_w = torch.ones(1, device=DEV)
    b = I.bias_normal(N, (912,)).to(DEV)
    y = F.fp8_linear(a, qw, s_w, b)
    torch.cuda.synchronize()
    assert torch.equal(y, b.expand(M, N))


def test_m_zero_is_noop():
    y = torch.full((0, 8), 1.0, dtype=torch.bfloat16, device=DEV)
    qw, s_w = F.fp8_quantize_weight(torch.ones((8, 32), dtype=torch.bfloat16, device=DEV))
    F.fp8_linear(torch.empty((0, 32), dtype=torch.bfloat16, device=DEV), qw, s_w, out=y)
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [8, 1000])
def test_linear_is_deterministic(M):
    K, N = 4096, 1024
    a = I.activations_normal(M, K, (913, M)).to(DEV)
    qw, s_w = F.fp8_quantize_weight(I.weights_normal(N, K, (914,)).to(DEV))
    y1 = F.fp8_linear(a, qw, s_w)
    y2 = F.fp8_linear(a, qw, s_w)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_back_to_back_layers_on_one_stream():
    """Each layer consumes the previous layer's output on one stream, so the programmatic
    dependent launches must order correctly: the chained result must equal the same layers
    run with a host synchronization between them. Layer 0 is also checked against the oracle."""
    K = 1024
    w = [I.weights_normal(K, K, (915, i)) for i in range(3)]
    q = [F.fp8_quantize_weight(x.to(DEV)) for x in w]
    torch.cuda.synchronize()
    for M in (4, 256):
        a0 = I.activations_normal(M, K, (916, M))
        x = a0.to(DEV)
        chained = []
        for qw, s_w in q:
            x = F.fp8_linear(x, qw, s_w)
            chained.append(x)
        torch.cuda.synchronize()
        x = a0.to(DEV)
        for i, (qw, s_w) in enumerate(q):
            x = F.fp8_linear(x, qw, s_w)
            torch.cuda.synchronize()
            assert torch.equal(x, chained[i]), f"M={M} layer {i}"
        linear_parity(chained[0], a0, w[0], False, what=f"chain M={M} layer 0")


@pytest.mark.parametrize("M,K", [(1, 4096), (5, 1000), (16, 4096), (16, 14336)])
def test_gemv_in_kernel_quantization_codes(M, K):
    """The decode GEMV quantizes A inside the kernel. With W = I (per-tensor: s_w = 1/448, code
    0x7E on the diagonal) each output is a single product, Y[m, n] = bf16(s_a * dec(qA[m, n])):
    neighbouring e4m3 codes differ by >= 12.5%, far beyond the tolerance, so every code the
    kernel chose is checked. Row 0 holds all positive e4m3 rounding midpoints and 448 with
    unit scale, where the quotient sits exactly on a rounding boundary."""
    from oracle import fp8_oracle as O
    g = np.random.default_rng(40 + M + K)
    a = (g.standard_normal((M, K)) * np.exp2(g.integers(-14, 9, (M, K)))).astype(np.float32)
    pos = np.array([O._decode_code(c) for c in range(0x7F)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    a[0, :] = 0.0
    a[0, :min(K, mids.size)] = mids[:K]
    a[0, -1] = 448.0
    if M > 1:
        a[1:] = np.clip(a[1:], -448, 448)
    a = I.to_bf16(a)
    w = torch.eye(K, dtype=torch.bfloat16)
    check(a, w, False, None, f"identity M={M} K={K}")


def test_pair_mode_needs_local_device_memory():
    """The two-SM pair GEMM is planned only for operands in this GPU's own memory; a pinned
    host buffer (reachable by the GPU) gets the single-CTA plan. Only the plan is queried:
    nothing is launched on host memory."""
    M, K, N = 512, 1024, 768
    qa = torch.zeros((M, K), dtype=torch.uint8, device=DEV)
    qw = torch.zeros((N, K), dtype=torch.uint8, device=DEV)
    cfg_dev = F.fp8_gemm_config(qa, qw)
    assert cfg_dev["two_sm"] and cfg_dev["grid"] % 2 == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for qa_x, qw_x in ((qa.cpu().pin_memory(), qw), (qa, qw.cpu().pin_memory())):
        cfg = F.fp8_gemm_config(qa_x, qw_x)
        assert not cfg["two_sm"] and 0 < cfg["grid"] <= sms
    # one row block: single CTA per tile as well
    assert not F.fp8_gemm_config(qa[:100], qw)["two_sm"]


@pytest.mark.parametrize("M,K,N", [(16384, 4096, 4096), (16384, 14336, 4096), (16384, 4096, 28672), (300, 4096, 512)])
def test_gemm_raster_groups(M, K, N):
    """Launch plan of the prefill layers: one raster group (all of W kept hot) when W fits the
    72 MB budget, else column groups of a ~28 MB W slice."""
    qa = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    qw = torch.empty((N, K), dtype=torch.uint8, device=DEV)
    cfg = F.fp8_gemm_config(qa, qw)
    n_tiles = (N + 255) // 256
    if N * K <= 72 << 20:
        assert cfg["group_n"] == n_tiles
    else:
        assert cfg["group_n"] == max(1, min(n_tiles, (28 << 20) // (256 * K)))


SPLIT_SHAPES = [(40, 5632, 5120), (48, 14336, 4096), (64, 8192, 4096), (100, 8192, 6144), (128, 5632, 2048),
                (33, 4100, 1027)]


@pytest.mark.parametrize("M,K,N", SPLIT_SHAPES)
def test_gemm_split_k(M, K, N):
    """Shapes with too few output tiles to fill the GPU split K across CTAs (fp32 partials in the
    workspace, reduced in split order by a second kernel): Y against the oracle, both scale
    modes with bias, guard bands intact, and the same bits on a second call."""
    assert not F.fp8_uses_gemv(M, K, N)
    a = I.activations_heavy_tail(M, K, (919, M, K))
    w = I.weights_row_std(N, K, (920, N, K))
    b = I.bias_normal(N, (921, N))
    qa = torch.zeros((M, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    qw = torch.zeros((N, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    cfg = F.fp8_gemm_config(qa, qw, K, F.fp8_workspace_bytes(M, K, N))
    assert cfg["splits"] > 1, cfg
    for pc in (False, True):
        check(a, w, pc, b, f"split-K {M}x{K}x{N} pc={pc}", check_w=False)
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=True)
    ad = a.to(DEV)
    y1 = F.fp8_linear_channelwise(ad, qw, s_w, b.to(DEV))
    y2 = F.fp8_linear_channelwise(ad, qw, s_w, b.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M", [100, 200])
@pytest.mark.parametrize("splits", [2, 3, 7, 16])
def test_gemm_forced_split_counts(M, splits, monkeypatch):
    """Split counts forced over the planner's range on a ragged K (17 blocks: a request is
    lowered until every split owns blocks), one CTA per tile (M = 100) and pairs with a partial
    second row block (M = 200), per-channel scales and bias."""
    monkeypatch.setenv("FP8W8A8_GEMM_SPLITK", str(splits))
    K, N = 2050, 777
    kb = (K + 127) // 128
    expect = -(-kb // -(-kb // splits))
    a = I.activations_heavy_tail(M, K, (922, splits))
    w = I.weights_row_std(N, K, (923,))
    b = I.bias_normal(N, (924,))
    qa = torch.zeros((M, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    qw = torch.zeros((N, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    cfg = F.fp8_gemm_config(qa, qw, K, F.fp8_workspace_bytes(M, K, N) + splits * M * 780 * 4)
    assert cfg["splits"] == expect and cfg["two_sm"] == (M > 128)
    ws = torch.empty(F.min_workspace_bytes(M, K, N) + 256 + 4096 + splits * M * 780 * 4, dtype=torch.uint8,
                     device=DEV)
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=True)
    buf, y, base, row_bytes, used = guarded((M, N), torch.bfloat16, DEV)
    F.fp8_linear_channelwise(a.to(DEV), qw, s_w, b.to(DEV), out=y, ws=ws)
    torch.cuda.synchronize()
    assert F.fp8_last_device_status() == F.FP8_OK
    assert_guards_intact(buf, base, row_bytes, used, M)
    linear_parity(y, a, w, True, b, what=f"forced split {splits}")


def test_gemm_split_k_strided_activations_and_odd_ldy():
    """K split with a strided A (TMA reads the padded rows) and an output whose row stride is
    odd (the reduce kernel's scalar stores): guard bands and the oracle's tolerance."""
    M, K, N = 40, 4100, 1027
    a = I.activations_heavy_tail(M, K, (928,))
    w = I.weights_row_std(N, K, (929,))
    b = I.bias_normal(N, (930,))
    qw, s_w = F.fp8_quantize_weight(w.to(DEV), per_channel=True)
    big = torch.zeros((M, K + 24), dtype=torch.bfloat16)
    big[:, :K] = a
    ad = big.to(DEV)[:, :K]
    ws = F.workspace(M, K, N, DEV)
    qa0 = torch.zeros((M, F.min_ld(K)), dtype=torch.uint8, device=DEV)
    assert F.fp8_gemm_config(qa0, qw, K, ws.numel())["splits"] > 1
    ybig = torch.full((M, N + 3), 7.0, dtype=torch.bfloat16, device=DEV)
    F.fp8_linear_channelwise(ad, qw, s_w, b.to(DEV), out=ybig[:, :N], ws=ws)
    torch.cuda.synchronize()
    assert F.fp8_last_device_status() == F.FP8_OK
    assert torch.all(ybig[:, N:] == 7.0)
    linear_parity(ybig[:, :N], a, w, True, b, what="split-K strided A, odd ldy")
