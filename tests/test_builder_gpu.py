"""Segment builder on the GPU against the oracle's stable sort: bit-exact."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _layer(S, T_max, K=64, N=64):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    W = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    layer = LoraLayer(W, S, 4, T_max)
    A = torch.zeros(K, 1, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, N, dtype=torch.bfloat16, device="cuda")
    for s in range(S):
        layer.load(s, A, B, 1.0)
    return layer


CASES = [
    ("one_row", 4, np.array([2])),
    ("one_base_row", 4, np.array([-1])),
    ("all_base", 8, np.full(300, -1)),
    ("all_one_slot", 8, np.full(1000, 5)),
    ("worked_example", 2, np.array([0, -1, 1, 0, 1, -1])),
    ("handbook_toy", 8, np.repeat([3, 5, 3, 0, 7, 5], [1, 1, 37, 1, 12, 1])),
    ("descending", 64, np.arange(63, -1, -1)),
]


def _random_cases():
    rng = np.random.default_rng(5)
    out = []
    for k, (T, S) in enumerate([(256, 128), (8192, 32), (4096, 100), (777, 3), (33, 1000),
                                (5000, 4096), (65536, 128), (1, 1), (31, 7), (1025, 64)]):
        ids = rng.integers(-1, S, size=T)
        out.append(("random_%d_T%d_S%d" % (k, T, S), S, ids))
    # long runs, as in prefill batches
    ids = np.repeat(rng.integers(-1, 50, size=40), rng.integers(1, 400, size=40))
    out.append(("runs", 50, ids))
    return out


@pytest.mark.parametrize("name,S,ids", CASES + _random_cases(), ids=lambda v: v if isinstance(v, str) else "")
def test_segments_bit_exact(name, S, ids):
    ids = ids.astype(np.int32)
    T = ids.shape[0]
    layer = _layer(S, T)
    layer.set_batch(torch.from_numpy(ids).cuda())
    perm, offs, sslot = layer.segments()
    ref_perm, ref_offs, ref_slot, bad = oracle.segments(ids, S)
    assert bad == 0
    assert np.array_equal(perm, ref_perm), name
    assert np.array_equal(offs, ref_offs), name
    assert np.array_equal(sslot, ref_slot), name
    assert layer.status() == 0
    layer.close()


def test_bad_and_empty_slot_ids_are_flagged_and_excluded():
    from segmented_rank_gemm_gb300.lora import LoraLayer, LORA_EID, LORA_OK
    S, K, N = 6, 64, 64
    W = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    layer = LoraLayer(W, S, 4, 32)
    A = torch.zeros(K, 1, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, N, dtype=torch.bfloat16, device="cuda")
    for s in (0, 1, 2, 4):  # slots 3 and 5 stay empty
        layer.load(s, A, B, 1.0)
    ids = np.array([0, 3, 7, -1, 2, -5, 4, 5, 1, 0], np.int32)
    layer.set_batch(torch.from_numpy(ids).cuda())
    perm, offs, sslot = layer.segments()
    assert layer.status() == LORA_EID
    assert layer.status() == LORA_OK  # flags were cleared
    clean = np.where(np.isin(ids, [0, 1, 2, 4]), ids, -1).astype(np.int32)
    ref_perm, ref_offs, ref_slot, _ = oracle.segments(clean, S)
    assert np.array_equal(perm, ref_perm) and np.array_equal(offs, ref_offs)
    assert np.array_equal(sslot, ref_slot)
    layer.close()
