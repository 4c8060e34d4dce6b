"""The oracle's composition evaluator (several adapters summed per row, with weights)
against what fixes it from outside:

- one member of weight 1 is the plain layer: equal to the C oracle's row-by-row evaluator;
- a composition is the base product plus the sum of its members' deltas, each member's
  delta taken from the C oracle with that member alone in a slot, times its weight;
- linearity in the weights: (a, w1) + (a, w2) equals (a, w1 + w2); all weights 0 give the
  base product;
- merged weight: a batch on one composed slot equals x (W + sum_m w_m (alpha_m / r_m) A_m B_m).

Mistaken copies (the scale over the summed rank, weights dropped, only the first member
kept -- the page warns that a composition is not identified by its first adapter) fail.
"""
import numpy as np
import pytest
import torch

import oracle


def _case(seed, T=23, K=24, N=20, ranks=(2, 5, 3, 1)):
    g = torch.Generator().manual_seed(seed)
    W = torch.randn(K, N, generator=g, dtype=torch.float64)
    x = torch.randn(T, K, generator=g, dtype=torch.float64)
    members = [(torch.randn(K, r, generator=g, dtype=torch.float64),
                torch.randn(r, N, generator=g, dtype=torch.float64), 2.0 * r + 1.0,
                float(w)) for r, w in zip(ranks, (0.5, -1.25, 2.0, 0.75))]
    return x, W, members


def _base(x, W):
    return x.numpy() @ W.numpy()


def pins(fn):
    x, W, m = _case(1)
    T, K = x.shape
    N = W.shape[1]
    rng = np.random.default_rng(2)
    ids = torch.tensor(rng.integers(-1, 3, size=T), dtype=torch.int32)
    # one member, weight 1: the plain layer (C oracle, row by row)
    plain = [(A, B, al) for A, B, al, _ in m[:3]]
    want = oracle.forward_rows(x, W, oracle.SlotTable(plain, K, N), ids)
    got = fn(x, W, [[(A, B, al, 1.0)] for A, B, al in plain], ids)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # base + sum of the members' deltas, each from the C oracle with that member alone
    comps = [m[:2], m[1:4], [m[0]]]
    got = fn(x, W, comps, ids)
    want = _base(x, W)
    for s, comp in enumerate(comps):
        for A, B, al, w in comp:
            alone = [None] * 3
            alone[s] = (A, B, al)
            d = oracle.forward_rows(x, W, oracle.SlotTable(alone, K, N), ids) - _base(x, W)
            want = want + w * d
    assert np.allclose(got, want, rtol=1e-11, atol=1e-11)
    # linearity in the weights, and all-zero weights
    A, B, al, _ = m[1]
    a = fn(x, W, [[(A, B, al, 0.25), (A, B, al, 1.5)]], ids)
    b = fn(x, W, [[(A, B, al, 1.75)]], ids)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    z = fn(x, W, [[(A, B, al, 0.0) for A, B, al, _ in m]], ids)
    assert np.array_equal(z, _base(x, W))
    # merged weight on a batch of one composed slot
    ones = torch.zeros(T, dtype=torch.int32)
    Wm = W.numpy().copy()
    for A, B, al, w in m:
        Wm += w * (al / A.shape[1]) * (A.numpy() @ B.numpy())
    assert np.allclose(fn(x, W, [m], ones), x.numpy() @ Wm, rtol=1e-10, atol=1e-10)
    return True


def test_composition_pins():
    assert pins(oracle.forward_composed)


def _summed_rank_scale(x, W, comps, slot):
    x, W, slot = x.numpy(), W.numpy(), slot.numpy()
    y = x @ W
    for s, comp in enumerate(comps):
        rows = np.nonzero(slot == s)[0]
        rs = sum(A.shape[1] for A, _, _, _ in comp)
        for A, B, al, w in comp:
            y[rows] += w * (al / rs) * ((x[rows] @ A.numpy()) @ B.numpy())
    return y


def _no_weight(x, W, comps, slot):
    return oracle.forward_composed(x, W, [[(A, B, al, 1.0) for A, B, al, _ in c] for c in comps],
                                   slot)


def _first_only(x, W, comps, slot):
    return oracle.forward_composed(x, W, [c[:1] for c in comps], slot)


@pytest.mark.parametrize("mutant", [_summed_rank_scale, _no_weight, _first_only])
def test_composition_pins_catch_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        pins(mutant)
