"""Every tiling of the tcgen05 base GEMM against the CPU oracle, element by element.

The automatic plan picks one tiling per batch shape, so a shape alone exercises only one
kernel variant.  Here the layer's plan is fixed through lora_set_gemm_plan to each N tile
(64 / 128 / 256), K split (1 / 2 / 4, delta mode only) and CTA pairing (cta_group::2), on
ragged shapes: row tiles with a partial last tile (and, for pairs, a last CTA wholly past
the batch), K ranges of unequal length, and N not a multiple of the tile."""
import pytest
import torch

from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, build_layer, oracle_rows, run_layer

pytestmark = pytest.mark.gpu

DELTA_PLANS = [(64, 1, 0), (64, 2, 0), (128, 1, 0), (128, 2, 0), (128, 4, 0), (256, 1, 0),
               (256, 2, 0), (256, 4, 0), (128, 1, 1), (128, 2, 1), (128, 4, 1), (256, 1, 1),
               (256, 2, 1), (256, 4, 1)]
V_PLANS = [(64, 1, 0), (128, 1, 0), (256, 1, 0), (128, 1, 1), (256, 1, 1)]


def _sweep(wl, plans):
    layer = build_layer(wl)
    ref = oracle_rows(wl)
    try:
        for bn, cs, pair in plans:
            layer.set_gemm_plan(bn, cs, pair)
            y = run_layer(layer, wl)
            assert layer.status() == 0, (bn, cs, pair)
            assert_parity(y, ref, wl.dtype, what="%s plan (%d, %d, %d)" % (wl.name, bn, cs, pair))
        layer.set_gemm_plan(0)
        assert_parity(run_layer(layer, wl), ref, wl.dtype, what=wl.name + " automatic plan")
    finally:
        layer.close()


def test_delta_mode_every_plan():
    # 3 row tiles (a pair's last CTA lies wholly past row 300), 17 K blocks (ranges 5/5/5/2
    # at a 4-way split), N = 1040 (a partial last tile for every N tile)
    wl = workloads.synthetic(4101, 300, 1032, 1040, S=9, ranks=[16, 1, 8, 16, 3, 12, 16, 5, 2],
                             R=16, base_frac=0.2)
    _sweep(wl, DELTA_PLANS)


def test_delta_mode_one_row_pairs():
    # a single row: a pair's second CTA has no rows at all (17 K blocks: every split valid)
    wl = workloads.synthetic(4102, 1, 1032, 264, S=3, ranks=8, R=8, base_frac=0.0)
    _sweep(wl, [(128, 2, 1), (256, 4, 1), (128, 1, 0)])


@pytest.mark.parametrize("T,K,N", [(512, 4096, 14336), (400, 1032, 14328), (300, 520, 10240)])
def test_delta_mode_automatic_plan_wide_n(T, K, N):
    # wide outputs on the automatic plan: where one tile per CTA (pair) would leave a last
    # round at most half full, the batch runs as two launches (the whole rounds' column
    # tiles, then the rest with a 2-way K split); ragged rows, K blocks and last tile
    wl = workloads.synthetic(4120 + T, T, K, N, S=7, ranks=[16, 4, 8, 16, 1, 12, 16], R=16,
                             base_frac=0.1)
    layer = build_layer(wl)
    try:
        for rep in range(2):
            y = run_layer(layer, wl)
            assert layer.status() == 0
            assert_parity(y, oracle_rows(wl), wl.dtype, what="%s automatic plan, launch %d" % (wl.name, rep))
    finally:
        layer.close()


def test_v_mode_every_plan():
    # 700 rows in 5.5 row tiles (pairs: 3 pairs, the last CTA partial), 9 K blocks,
    # N = 1000; many slots per tile so every tile runs several expand blocks
    wl = workloads.synthetic(4103, 700, 520, 1000, S=24, ranks=16, R=16, base_frac=0.1,
                             layout="runs")
    _sweep(wl, V_PLANS)


def test_v_mode_stream_k_tail():
    # more tiles than resident CTAs (pairs), with a short last round: on 152 SMs every
    # tiling below leaves 12 to 64 tiles over, which are cut in two (head and tail on two
    # CTAs, the tail added to the head's accumulator as an fp32 partial); 17 K blocks give
    # halves of 8 and 9
    wl = workloads.synthetic(4106, 2600, 1032, 2048, S=24, ranks=16, R=16, base_frac=0.1,
                             layout="runs")
    _sweep(wl, [(256, 1, 0), (128, 1, 0), (64, 1, 0), (256, 1, 1), (128, 1, 1)])


def test_v_mode_wide_rank_pairs():
    # rank 64: two expand blocks per slot (hi and lo halves in separate blocks)
    wl = workloads.synthetic(4104, 900, 384, 512, S=10, ranks=[64, 40, 8, 64, 17, 64, 1, 33, 64, 2],
                             R=64, base_frac=0.05, layout="random")
    _sweep(wl, [(128, 1, 1), (256, 1, 1), (256, 1, 0)])


def test_invalid_plans_rejected():
    from segmented_rank_gemm_gb300.lora import LoraError
    wl = workloads.synthetic(4105, 8, 64, 64, S=2, ranks=4, R=8)
    layer = build_layer(wl)
    try:
        for bad in [(96, 1, 0), (64, 4, 0), (64, 1, 1), (128, 3, 0), (256, 8, 0), (128, 1, 2)]:
            with pytest.raises(LoraError):
                layer.set_gemm_plan(*bad)
        # a K split with an empty K range fails at forward time, not silently
        layer.set_gemm_plan(128, 4, 0)  # K = 64: one K block cannot be split four ways
        with pytest.raises(LoraError):
            run_layer(layer, wl)
    finally:
        layer.close()
