"""Batches of more than 512 bf16 rows (the prefill regime: tensor-core SGMV shrink into v,
then the base GEMM with the expand of v) against the CPU oracle, element by element:
ragged K and N, slot rank widths that are not multiples of 16, full rank 128, one segment
spanning many 128-row tiles, many short segments, empty slots and base-only rows, and the
same layer reused across batches of different sizes."""
import pytest
import torch

from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, build_layer, oracle_rows, run_layer

pytestmark = pytest.mark.gpu


def _check(wl, **kw):
    layer = build_layer(wl, **kw)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), wl.dtype, what=wl.name)
    layer.close()


CASES = [
    # T, K, N, S, ranks, R, layout, base_frac
    (600, 520, 264, 5, [8, 16, 3, 12, 1], 16, "runs", 0.2),     # K, N not tile multiples
    (1000, 256, 384, 7, 8, 8, "random", 0.1),                   # rank width 8 < MMA N 16
    (777, 384, 200, 3, [24, 5, 17], 24, "sorted", 0.1),         # width 24 -> MMA N 32
    (1100, 512, 512, 4, [1, 128, 64, 7], 128, "runs", 0.1),     # width 128
    (2000, 1024, 256, 40, 64, 64, "random", 0.05),              # 40 segments, width 64
    (1300, 256, 256, 1, 16, 16, "random", 0.0),                 # one segment, 11 tiles
]


@pytest.mark.parametrize("T,K,N,S,ranks,R,layout,base", CASES)
def test_vmode_shapes(T, K, N, S, ranks, R, layout, base):
    wl = workloads.synthetic(400 + T, T, K, N, S=S, ranks=ranks, R=R, layout=layout,
                             base_frac=base)
    _check(wl)


def test_vmode_empty_slots_and_base_rows():
    wl = workloads.synthetic(410, 700, 256, 256, S=5, ranks=8, R=8, base_frac=0.1,
                             empty_slots=(1, 3))
    _check(wl)


def test_vmode_all_base_only():
    wl = workloads.synthetic(411, 600, 256, 128, S=3, ranks=16, R=16, base_frac=1.0)
    _check(wl)


def test_vmode_layer_reused_across_batches():
    big = workloads.synthetic(412, 1500, 256, 256, S=6, ranks=[16, 8, 4, 16, 2, 9], R=16,
                              base_frac=0.1, layout="runs")
    layer = build_layer(big, max_tokens=1500)
    for T in (1500, 700, 513, 1024):
        wl = workloads.synthetic(412, T, 256, 256, S=6, ranks=[16, 8, 4, 16, 2, 9], R=16,
                                 base_frac=0.1, layout="random")
        # same seed, same weights and adapters: only the batch differs
        assert torch.equal(wl.W, big.W)
        y = run_layer(layer, wl)
        assert layer.status() == 0
        assert_parity(y, oracle_rows(wl), wl.dtype, what="T=%d" % T)
    layer.close()
