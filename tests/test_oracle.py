"""The CPU oracle against its pins (page-printed values, library special cases,
closed forms, invariants, brute force) and the pages' size arithmetic."""
import numpy as np
import pytest

import oracle
from oracle import sizes
import oracle_pins
from oracle_pins import golden


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.lib())


def test_p1_worked_memory_example():
    g = golden("adapter_sizes.json")
    attn4 = [(4096, 4096)] * 4
    assert sizes.adapter_params([(4096, 4096)], 16) == g["p1_per_projection"]
    assert sizes.adapter_params(attn4, 16) == g["p1_per_layer"]
    total = sizes.adapter_params(attn4, 16, layers=32)
    assert total == g["p1_total_params"]
    assert abs(total * 2 / 1e6 - g["p1_total_mb"]) < 0.1  # 33,554,432 B
    # every linear layer (attention at 4096 x 4096 plus the three MLP projections)
    all_lin = attn4 + [(4096, 14336), (4096, 14336), (14336, 4096)]
    mb = sizes.adapter_bytes(all_lin, 16, layers=32) / 1e6
    assert abs(mb - g["p1_all_linear_mb_approx"]) / g["p1_all_linear_mb_approx"] < 0.05


def test_p2_eighty_mb_adapter_and_hundred_resident():
    g = golden("adapter_sizes.json")
    shapes = list(sizes.LLAMA8B_PROJECTIONS.values())
    nbytes = sizes.adapter_bytes(shapes, 16, layers=32)
    assert nbytes == 83_886_080  # exactly 80 MiB
    assert abs(nbytes / 2**20 - g["p2_all7_rank16_mb_approx"]) < 1e-9
    resident = 8 * 2**30 / nbytes
    assert abs(resident - g["p2_resident_in_8gb_approx"]) / 100 < 0.05
    share = sizes.lora_flop_share(shapes, 16)
    assert 0.5 * g["p2_compute_share_approx"] < share < 2 * g["p2_compute_share_approx"]


def test_p3_capacity_example():
    g = golden("adapter_sizes.json")
    p = sizes.LLAMA8B_PROJECTIONS
    attn = [p["q"], p["k"], p["v"], p["o"]]
    per_adapter = sizes.adapter_bytes(attn, 16, layers=32)
    lo_gb, hi_gb = g["p3_reservation_gb_range"]
    lo_fit, hi_fit = lo_gb * 1e9 / per_adapter, hi_gb * 1e9 / per_adapter
    want_lo, want_hi = g["p3_attention_rank16_fit_range"]
    assert abs(lo_fit - want_lo) / want_lo < 0.1 and abs(hi_fit - want_hi) / want_hi < 0.1
    params64 = sizes.adapter_params(list(p.values()), 64, layers=32)
    assert abs(params64 / 1e6 - g["p3_all7_rank64_params_m_approx"]) < 1
    assert abs(params64 * 2 / 1e6 - g["p3_all7_rank64_mb_approx"]) < 1
    fit = hi_gb * 1e9 / (params64 * 2)
    assert abs(fit - g["p3_all7_rank64_fit_approx"]) <= 5


def test_oracle_is_fp64_and_threads():
    assert oracle.num_threads() >= 1
    wl_x = np.ones((2, 3))
    t = oracle.SlotTable([None], 3, 2)
    y = oracle.forward_rows(wl_x, np.ones((3, 2)) / 3, t, np.array([-1, -1], np.int32))
    assert y.dtype == np.float64 and np.all(y == 1.0)
