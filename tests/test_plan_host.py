"""The GEMM launch planner on the host (fp8_gemm_plan_model: the rules fp8_gemm_config reports on a
GPU, evaluated without one) for a 152-SM GB300 with 76 co-resident CTA pairs: pair mode, raster
groups, the column split of the last wave or of every tile, and the K split."""

import pytest

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I

SMS, PAIRS = 152, 76
L2_BUDGET = 72 << 20          # W kept hot in L2 up to this many bytes
W_SLICE = 28 << 20            # else column groups of about this many bytes of W


@pytest.fixture(scope="module", autouse=True)
def lib():
    F.lib()


def plan(M, N, K, ws=None, sms=SMS, pairs=PAIRS):
    ws = F.fp8_workspace_bytes(M, K, N) if ws is None else ws
    return F.fp8_gemm_plan_model(M, N, K, sms, pairs, ws)


def tiles(M, N, two):
    m_units = -(-M // 256) if two else -(-M // 128)
    return m_units * -(-N // 256)


@pytest.mark.parametrize("layer", range(4))
def test_prefill_layers(layer):
    """Llama-3-8B linears at M = 16384: CTA pairs on all 152 SMs, no K split, W kept hot when it
    fits the budget (else ~28 MB column groups), and the partial last wave in 128-column halves."""
    L = I.LLAMA8B_LAYERS[layer]
    p = plan(16384, L.N, L.K)
    assert p["two_sm"] and p["grid"] == SMS and p["splits"] == 1
    n_tiles = -(-L.N // 256)
    w_bytes = L.N * F.min_ld(L.K)
    assert p["group_n"] == (n_tiles if w_bytes <= L2_BUDGET else max(1, min(n_tiles, W_SLICE // (256 * L.K))))
    units = tiles(16384, L.N, True)
    rem = units % PAIRS
    assert rem > 0 and 2 * rem <= PAIRS and p["tail_split"] == 2


def test_last_wave_split_only_when_it_fits_one_wave():
    """The last wave is split only when its tiles, halved, fit the pairs; whole waves stay whole."""
    N, K = 2560, 512                                  # 10 column tiles
    for m_units, expect in ((8, 2), (10, 2), (12, 1), (76, 1)):
        # 80 units: 4 left (halves fit); 100: 24 left (48 <= 76); 120: 44 left (88 > 76); 760: whole waves
        p = plan(m_units * 256, N, K)
        assert p["two_sm"] and p["grid"] == SMS
        assert p["tail_split"] == expect, (m_units, p)


@pytest.mark.parametrize("M,N,K,two,f", [(33, 2560, 2048, False, 4), (100, 2560, 2048, False, 4),
                                         (64, 4096, 4096, False, 4), (64, 11264, 2048, False, 2),
                                         (300, 1027, 1000, True, 4), (257, 3001, 2050, True, 2)])
def test_small_m_column_split(M, N, K, two, f):
    """Few tiles and at most 32 K blocks: no K split; every tile split into 4 units where four
    times the tiles fit the slots, else 2; the grid is one CTA (pair) per unit."""
    p = plan(M, N, K)
    assert p["two_sm"] == two and p["splits"] == 1 and p["tail_split"] == f, p
    units = tiles(M, N, two) * f
    assert p["grid"] == (2 * units if two else units)


@pytest.mark.parametrize("M,N,K", [(64, 4096, 14336), (128, 2048, 5632), (33, 1027, 4100), (48, 4096, 14336)])
def test_small_m_long_k_splits_k(M, N, K):
    """More than 32 K blocks on one row block: the K split (fp32 partials in the workspace), never
    combined with a column split; without room for the partials, neither."""
    p = plan(M, N, K)
    assert not p["two_sm"] and p["splits"] > 1 and p["tail_split"] == 1, p
    assert p["grid"] <= SMS
    q = plan(M, N, K, ws=F.min_workspace_bytes(M, K, N))
    assert q["splits"] == 1


def test_pair_mode_needs_enough_pairs():
    """Pairs only with at least two row blocks and pairs on 3/4 of the SMs; otherwise one CTA
    per tile (and a K split may come back)."""
    assert plan(256, 4096, 4096)["two_sm"]
    assert not plan(128, 4096, 4096)["two_sm"]
    assert not plan(16384, 4096, 4096, pairs=0)["two_sm"]
    assert not plan(16384, 4096, 4096, pairs=56)["two_sm"]   # 112 of 152 SMs < 3/4
    assert plan(16384, 4096, 4096, pairs=57)["two_sm"]


def test_grid_never_exceeds_the_gpu():
    for M in (33, 129, 256, 1000, 4096, 16384):
        for N in (256, 1027, 4096, 28672):
            for K in (128, 2048, 14336):
                p = plan(M, N, K)
                assert 0 < p["grid"] <= SMS and (p["grid"] % 2 == 0 or not p["two_sm"]), (M, N, K, p)
                assert p["splits"] == 1 or p["tail_split"] == 1


def test_plan_model_rejects_bad_sizes():
    for args in ((0, 4096, 4096, SMS, PAIRS, 0), (16, 0, 4096, SMS, PAIRS, 0), (16, 4096, 0, SMS, PAIRS, 0),
                 (16, 4096, 4096, 0, PAIRS, 0), (16, 4096, 4096, SMS, -1, 0)):
        with pytest.raises(F.FP8Error):
            F.fp8_gemm_plan_model(*args)
