"""Full-size workloads on the GPU, in the launch configuration the benchmark times,
against the oracle on every row: decode (256 rows), prefill (8192 rows in 32 segments)
and the continuous batch (4096 rows).  Every 128-row tile of the base GEMM, every
stream-K tail tile of its last round and every segment boundary is thereby covered."""
import numpy as np
import pytest

from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, build_layer, oracle_rows, run_layer

pytestmark = pytest.mark.gpu


def test_decode_bgmv_full():
    wl = workloads.decode_bgmv()
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), wl.dtype, what="decode_bgmv")
    # the segment layout of the batch is the oracle's, bit for bit
    import oracle
    perm, offs, sslot = layer.segments()
    rp, ro, rs, _ = oracle.segments(wl.token_slot, wl.S)
    assert np.array_equal(perm, rp) and np.array_equal(offs, ro) and np.array_equal(sslot, rs)
    layer.close()


def test_prefill_sgmv_every_row():
    wl = workloads.prefill_sgmv()
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), wl.dtype, what="prefill_sgmv")
    layer.close()


def test_mixed_continuous_every_row():
    wl = workloads.mixed_continuous()
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), wl.dtype, what="mixed_continuous")
    layer.close()
