"""The decode GEMV's launch configuration on the host (fp8_gemv_plan_model: the search the library
runs before every GEMV launch, with the device facts given): a configuration exists for the
decode layers the pages and the benchmark use, and it keeps the kernel's own invariants."""

import pytest

import fp8_w8a8_quantized_dynamic_gb300 as F
from fp8_w8a8_quantized_dynamic_gb300 import inputs as I

SMS = 152
# co-resident clusters of 1..8 CTAs (one CTA per SM at the GEMV's shared memory), shaped like a
# GB300's: clusters must fit inside a GPC, so larger clusters leave a few SMs unused
OCC = [148, 74, 48, 36, 28, 24, 20, 16]
SMEM = 227 * 1024
LAYERS = list(I.LLAMA8B_LAYERS) + list(I.TINYLLAMA_LAYERS)


@pytest.fixture(scope="module", autouse=True)
def lib():
    F.lib()


def check_invariants(cfg, M, N, K, mode):
    kt = -(-K // 128)
    S, C = cfg["cluster"], cfg["clusters"]
    assert 1 <= S <= 8 and 1 <= C <= OCC[S - 1] and S * C <= SMS
    slice_tiles = -(-kt // S)
    assert -(-kt // slice_tiles) == S                 # every rank of a cluster owns K tiles
    assert cfg["kslice"] == slice_tiles * 128 and cfg["kslice"] <= 4096
    row_blocks = -(-N // 128)
    assert -(-row_blocks // C) <= 8                   # row blocks per cluster fit the partials
    assert C == -(-row_blocks // -(-row_blocks // C))  # no cluster without row blocks
    assert 4 <= cfg["stages"] <= 12
    assert cfg["tcgen05"] == (1 if (M >= 17 and mode == 0) else 0)


@pytest.mark.parametrize("L", LAYERS, ids=[f"{L.name}{L.K}x{L.N}" for L in LAYERS])
def test_decode_layers_have_a_configuration(L):
    """Up to 16 tokens quantizing A in the kernel (bulk-copied into idle ring stages: A's rows
    are aligned), 17-32 tokens on activations quantized beforehand (tcgen05 main loop)."""
    for M in (1, 2, 4, 8, 15, 16):
        cfg = F.fp8_gemv_plan_model(M, L.N, L.K, 1, OCC, SMEM)
        check_invariants(cfg, M, L.N, L.K, 1)
        assert cfg["scratch_a"] in (1, 2)
        if cfg["scratch_a"] == 1:  # all of A in shared memory: every CTA takes the maximum itself
            assert cfg["cluster_amax"] == 0
    for M in (17, 24, 32):
        cfg = F.fp8_gemv_plan_model(M, L.N, L.K, 0, OCC, SMEM)
        check_invariants(cfg, M, L.N, L.K, 0)
        assert cfg["scratch_a"] == 0


def test_static_scale_copies_only_the_slice():
    """A static scale needs no maximum over A: at most the CTA's own slice is staged."""
    for L in I.LLAMA8B_LAYERS:
        cfg = F.fp8_gemv_plan_model(8, L.N, L.K, 1, OCC, SMEM, static_scale=True)
        assert cfg["scratch_a"] in (0, 2)


def test_weight_only_long_k():
    """bf16 activations: K up to 32768 (eight ranks of 4096 elements)."""
    cfg = F.fp8_gemv_plan_model(1, 4096, 32768, 2, OCC, SMEM)
    assert cfg["cluster"] == 8 and cfg["kslice"] == 4096 and cfg["tcgen05"] == 0


def test_more_clusters_never_stream_more_tiles_per_cta():
    """Doubling the co-resident clusters cannot make the busiest CTA stream more weight tiles (with
    fewer clusters a configuration may not exist at all: more row blocks per cluster hold more
    partials than shared memory takes)."""
    compared = 0
    for L in I.LLAMA8B_LAYERS:
        for M, mode in ((1, 1), (32, 0)):
            big = F.fp8_gemv_plan_model(M, L.N, L.K, mode, OCC, SMEM)
            try:
                small = F.fp8_gemv_plan_model(M, L.N, L.K, mode, [max(1, o // 2) for o in OCC], SMEM)
            except F.FP8Error as e:
                assert e.status == F.FP8_ERR_CUDA
                continue
            compared += 1

            def busiest(c):
                return -(-(-(-L.N // 128)) // c["clusters"]) * (c["kslice"] // 128)

            assert busiest(big) <= busiest(small)
    assert compared >= 4


def test_no_configuration_and_bad_arguments():
    # 32 tokens quantized in the kernel on a 14336 x 14336 weight: the activation area and the
    # partials leave no room for the ring (the library takes the pre-quantized path there)
    with pytest.raises(F.FP8Error) as e:
        F.fp8_gemv_plan_model(32, 14336, 14336, 1, OCC, SMEM)
    assert e.value.status == F.FP8_ERR_CUDA
    F.fp8_gemv_plan_model(32, 14336, 14336, 0, OCC, SMEM)
    for args in ((0, 4096, 4096, 1), (33, 4096, 4096, 0), (1, 4096, 40000, 1), (1, 0, 4096, 1), (1, 4096, 4096, 3)):
        with pytest.raises(F.FP8Error) as e:
            F.fp8_gemv_plan_model(*args, OCC, SMEM)
        assert e.value.status == F.FP8_ERR_INVALID_ARG
