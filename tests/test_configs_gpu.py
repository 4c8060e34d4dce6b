"""Full-size workloads on the GPU, in the launch configuration the benchmark times,
against the oracle on every row (decode) or on sampled rows that include the first and
last row of every segment (prefill, continuous batch)."""
import numpy as np
import pytest
import torch

from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, build_layer, oracle_rows, run_layer

pytestmark = pytest.mark.gpu


def _segment_edge_rows(ids, extra, seed):
    ids = np.asarray(ids)
    edges = [0, len(ids) - 1]
    change = np.nonzero(ids[1:] != ids[:-1])[0]
    edges += list(change) + list(change + 1)
    rng = np.random.default_rng(seed)
    edges += list(rng.choice(len(ids), size=extra, replace=False))
    return np.unique(np.asarray(edges, dtype=np.int64))


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


def test_prefill_sgmv_sampled():
    wl = workloads.prefill_sgmv()
    rows = _segment_edge_rows(wl.token_slot.numpy(), 32, 3)
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y[torch.from_numpy(rows).cuda()], oracle_rows(wl, rows), wl.dtype,
                  what="prefill_sgmv")
    layer.close()


def test_mixed_continuous_sampled():
    wl = workloads.mixed_continuous()
    rows = _segment_edge_rows(wl.token_slot.numpy(), 48, 4)
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == 0
    assert_parity(y[torch.from_numpy(rows).cuda()], oracle_rows(wl, rows), wl.dtype,
                  what="mixed_continuous")
    layer.close()
