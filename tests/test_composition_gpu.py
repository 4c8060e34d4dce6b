"""Composed slots on the GPU, through the C ABI (load_adapter_slot_composed), against the
oracle's composition evaluator: every kernel path that applies the slot scales -- the
decode BGMV (slot width <= 32 and wider), the tensor-core SGMV shrink of large batches,
and the fp32 tile kernel -- with compositions of 1 to 3 members, mixed ranks, negative and
zero weights, a member repeated, plain slots and an empty slot in the same batch.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def _members(g, K, N, ranks, weights, dtype, std):
    return [((torch.randn(K, r, generator=g) * std).to(dtype),
             (torch.randn(r, N, generator=g) * std).to(dtype), 2.0 * r, float(w))
            for r, w in zip(ranks, weights)]


def _run(seed, T, K, N, max_rank, dtype, recipes):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    g = torch.Generator().manual_seed(seed)
    std = 0.02
    W = (torch.randn(K, N, generator=g) * std).to(dtype)
    x = torch.randn(T, K, generator=g).to(dtype)
    comps = []
    for ranks, weights in recipes:
        comps.append(_members(g, K, N, ranks, weights, dtype, std) if ranks else None)
    # a member repeated inside one composition (the same adapter twice)
    if comps[0]:
        comps[0] = comps[0] + [(comps[0][0][0], comps[0][0][1], comps[0][0][2], -0.3)]
    S = len(comps)
    layer = LoraLayer(W.cuda(), S, max_rank, T)
    for s, comp in enumerate(comps):
        if comp is None:
            continue
        layer.load_composed(s, [(A.cuda(), B.cuda(), al, w) for A, B, al, w in comp])
    rng = np.random.default_rng(seed)
    ids = torch.tensor(rng.integers(-1, S, size=T), dtype=torch.int32)
    y = layer(x.cuda(), ids.cuda())
    torch.cuda.synchronize()
    empty = [s for s, c in enumerate(comps) if c is None]
    status = layer.status()
    assert status == (-4 if any(int(i) in empty for i in ids) else 0)
    ref = oracle.forward_composed(x, W, comps, ids)
    layer.close()
    return y, ref


RECIPES = [((4, 8), (0.5, 1.5)), ((16,), (1.0,)), ((1, 2, 5), (1.0, -0.7, 2.0)), (None, None),
           ((3, 3), (0.0, 1.0))]


@pytest.mark.parametrize("T", [300, 700])  # decode (BGMV) and prefill (tensor-core SGMV)
def test_compositions_bf16(T):
    y, ref = _run(10 + T, T, 256, 192, 16, BF16, RECIPES)
    assert_parity(y, ref, BF16, what="compositions, T=%d" % T)


@pytest.mark.parametrize("T", [200, 600])
def test_compositions_wide_slots_bf16(T):
    """Slot width 64: the row-major BGMV in decode, two K blocks of expand in prefill."""
    recipes = [((16, 24), (1.0, 0.5)), ((40, 8, 16), (0.25, -1.0, 1.0)), ((64,), (1.0,))]
    y, ref = _run(20 + T, T, 384, 200, 64, BF16, recipes)
    assert_parity(y, ref, BF16, what="wide compositions, T=%d" % T)


def test_compositions_fp32():
    y, ref = _run(30, 150, 72, 40, 16, F32, RECIPES)
    assert_parity(y, ref, F32, what="fp32 compositions")


def test_composition_rank_limits():
    from segmented_rank_gemm_gb300.lora import LoraError, LoraLayer
    g = torch.Generator().manual_seed(1)
    layer = LoraLayer(torch.zeros(64, 64, dtype=BF16, device="cuda"), 2, 16, 8)
    m = _members(g, 64, 64, (8, 9), (1.0, 1.0), BF16, 0.02)
    with pytest.raises(LoraError) as e:  # 8 + 9 > max_rank 16
        layer.load_composed(0, [(A.cuda(), B.cuda(), al, w) for A, B, al, w in m])
    assert e.value.code == -3
    with pytest.raises(LoraError):
        layer.load_composed(0, [])
    layer.close()
