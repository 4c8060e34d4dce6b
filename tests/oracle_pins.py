"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``pin_*`` function takes the bound oracle library (the real one, or a copy with a
planted mistake) and raises AssertionError when the oracle disagrees with:
  - values the pages print (segment counts, group sizes, element counts),
  - special cases that reduce to a library routine (numpy matmul of x W, of the merged
    weight W + (alpha/r) A B -- the merged-weight equivalence the pages state),
  - closed forms (rank 1 with a unit-vector A),
  - invariants (row permutation, slot relabelling, linearity in alpha, ignored padding),
  - brute force on tiny inputs (Python's stable ``sorted`` for the segment builder;
    exact integer arithmetic for the layer).
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np

import oracle
from segmented_rank_gemm_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def close(a, b, rel=1e-12):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b) / (1.0 + np.abs(b))
    assert err.size == 0 or float(err.max()) <= rel, float(err.max())


def all_evaluators(L, x, W, table, ids):
    rows = oracle.forward_rows(x, W, table, ids, _lib=L)
    grouped = oracle.forward_grouped(x, W, table, ids, _lib=L)
    merged = oracle.forward_merged(x, W, table, ids, _lib=L)
    return rows, grouped, merged


def rand_case(seed, T=24, K=20, N=12, S=4, ranks=(3, 1, 4, 2), base_frac=0.25):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((K, N))
    adapters = [(rng.standard_normal((K, r)), rng.standard_normal((r, N)),
                 float(rng.integers(1, 9))) for r in ranks[:S]]
    ids = rng.integers(0, S, size=T)
    ids[rng.random(T) < base_frac] = -1
    return x, W, adapters, ids.astype(np.int32)


# --------------------------------------------------------------------------------
# Page-printed values
# --------------------------------------------------------------------------------

def pin_worked_example_structure(L):
    """Six rows [finance, base, code, finance, code, base]: each group holds 2 rows;
    per-adapter delta 26 elements vs 40 for the full weight."""
    g = golden("worked_example.json")
    wl = workloads.worked_example()
    perm, offs, sslot, bad = oracle.segments(wl.token_slot, wl.S, _lib=L)
    assert bad == 0
    assert perm.tolist() == g["perm"] and offs.tolist() == g["seg_offsets"]
    assert sslot.tolist() == g["seg_slot"]
    sizes = {"base": int((wl.token_slot.numpy() == -1).sum())}
    for name, s in (("finance", 0), ("code", 1)):
        sizes[name] = int(offs[list(sslot).index(s) + 1] - offs[list(sslot).index(s)])
    assert sizes == g["grouped_batch_sizes"], sizes
    K, N, r = 8, 5, 2
    assert oracle.adapter_params([(K, N)], r) == g["per_adapter_delta_elements"]
    assert K * N == g["full_weight_elements"]


def pin_worked_example_values(L):
    """Grouped == per-row == merged, and each within the page's assert_close
    tolerance (1e-5) of a float32 evaluation by library matmul."""
    g = golden("worked_example.json")
    wl = workloads.worked_example()
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    rows, grouped, merged = all_evaluators(L, wl.x, wl.W, table, wl.token_slot)
    close(grouped, rows)
    close(merged, rows)
    # float32 library evaluation, group by group, as x times the merged weight
    x, W = wl.x.numpy(), wl.W.numpy()
    ref = np.zeros((wl.T, wl.N), dtype=np.float32)
    ids = wl.token_slot.numpy()
    for i in range(wl.T):
        if ids[i] < 0:
            ref[i] = x[i] @ W
        else:
            A, B, alpha = wl.adapters[ids[i]]
            Wm = W + (alpha / A.shape[1]) * (A.numpy() @ B.numpy())
            ref[i] = x[i] @ Wm
    tol = g["assert_close_rtol_atol"]
    assert np.all(np.abs(rows - ref) <= tol + tol * np.abs(ref)), np.abs(rows - ref).max()


def pin_handbook_toy(L):
    """53 rows, 6 requests, 4 SGMV segments (adapters {0,3,5,7}); the segment of each
    adapter holds the rows of its requests in their original order."""
    g = golden("handbook_toy.json")
    wl = workloads.handbook_toy()
    assert wl.T == g["rows"] and len(g["lengths"]) == g["requests"]
    perm, offs, sslot, bad = oracle.segments(wl.token_slot, wl.S, _lib=L)
    assert bad == 0 and len(sslot) == g["segments"]
    assert sslot.tolist() == sorted(set(g["owners"]))
    starts = np.cumsum([0] + g["lengths"][:-1])
    for s in sslot:
        expect = [int(starts[q]) + t for q, a in enumerate(g["owners"]) if a == s
                  for t in range(g["lengths"][q])]
        k = list(sslot).index(s)
        assert perm[offs[k]:offs[k + 1]].tolist() == expect
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    rows, grouped, merged = all_evaluators(L, wl.x, wl.W, table, wl.token_slot)
    close(grouped, rows)
    close(merged, rows)
    # the page's own check, restated: a library evaluation in fp32, one request at a time
    # (its rows times W, plus the scale times (rows A) B of its adapter), agrees with the
    # oracle at the printed tolerance (allclose, atol 1e-5)
    import torch
    parts, s0 = [], 0
    for a, n in zip(g["owners"], g["lengths"]):
        xr = wl.x[s0:s0 + n].float()
        A, B, alpha = wl.adapters[a]
        scale = alpha / A.shape[1]
        parts.append(torch.matmul(xr, wl.W.float()) +
                     scale * torch.matmul(torch.matmul(xr, A.float()), B.float()))
        s0 += n
    per_request = torch.cat(parts)
    assert torch.allclose(torch.from_numpy(np.asarray(rows)).float(), per_request,
                          atol=g["allclose_atol"])


# --------------------------------------------------------------------------------
# Special cases that reduce to a library routine
# --------------------------------------------------------------------------------

def pin_base_only_is_library_matmul(L):
    x, W, adapters, ids = rand_case(11)
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    ref = x @ W
    for out in all_evaluators(L, x, W, table, np.full(x.shape[0], -1, np.int32)):
        close(out, ref)
    # base rows of a mixed batch too
    for out in all_evaluators(L, x, W, table, ids):
        close(out[ids == -1], ref[ids == -1])


def pin_single_adapter_is_merged_library_matmul(L):
    """Every row on one adapter: y = x (W + (alpha/r) A B), numpy fp64."""
    x, W, adapters, _ = rand_case(12)
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    for s, (A, B, alpha) in enumerate(adapters):
        ref = x @ (W + (alpha / A.shape[1]) * (A @ B))
        for out in all_evaluators(L, x, W, table, np.full(x.shape[0], s, np.int32)):
            close(out, ref)


def pin_mixed_rows_are_merged_library_matmul(L):
    """A mixed batch: each adapted row equals x_i times its adapter's merged weight."""
    x, W, adapters, ids = rand_case(13, T=40)
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    ref = np.empty((x.shape[0], W.shape[1]))
    for i, s in enumerate(ids):
        if s < 0:
            ref[i] = x[i] @ W
        else:
            A, B, alpha = adapters[s]
            ref[i] = x[i] @ (W + (alpha / A.shape[1]) * (A @ B))
    for out in all_evaluators(L, x, W, table, ids):
        close(out, ref)


# --------------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------------

def pin_rank1_unit_vector(L):
    """Rank 1, A = e_k, B = b: y = x W + alpha * x[:, k] b."""
    rng = np.random.default_rng(14)
    T, K, N = 9, 7, 6
    x, W = rng.standard_normal((T, K)), rng.standard_normal((K, N))
    for k in (0, 3, K - 1):
        A = np.zeros((K, 1))
        A[k, 0] = 1.0
        b = rng.standard_normal((1, N))
        table = oracle.SlotTable([(A, b, 3.0)], K, N)
        ids = np.zeros(T, np.int32)
        ref = x @ W + 3.0 * np.outer(x[:, k], b[0])
        for out in all_evaluators(L, x, W, table, ids):
            close(out, ref)


def pin_zero_alpha_or_zero_B(L):
    x, W, adapters, ids = rand_case(15)
    base = x @ W
    zero_alpha = [(A, B, 0.0) for A, B, _ in adapters]
    zero_b = [(A, np.zeros_like(B), a) for A, B, a in adapters]
    for ads in (zero_alpha, zero_b):
        table = oracle.SlotTable(ads, W.shape[0], W.shape[1])
        for out in all_evaluators(L, x, W, table, ids):
            close(out, base)


def pin_linear_in_alpha(L):
    """Doubling alpha doubles each row's delta."""
    x, W, adapters, ids = rand_case(16)
    base = x @ W
    t1 = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    t2 = oracle.SlotTable([(A, B, 2 * a) for A, B, a in adapters], W.shape[0], W.shape[1])
    for f in (oracle.forward_rows, oracle.forward_grouped, oracle.forward_merged):
        d1 = f(x, W, t1, ids, _lib=L) - base
        d2 = f(x, W, t2, ids, _lib=L) - base
        close(d2, 2 * d1, rel=1e-10)
        assert np.abs(d1[ids >= 0]).max() > 1e-3  # adapted rows really carry a delta


def pin_row_permutation(L):
    """Permuting rows together with their ids permutes y (bit for bit)."""
    x, W, adapters, ids = rand_case(17, T=30)
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    p = np.random.default_rng(170).permutation(x.shape[0])
    for f in (oracle.forward_rows, oracle.forward_grouped, oracle.forward_merged):
        y = f(x, W, table, ids, _lib=L)
        yp = f(x[p], W, table, ids[p], _lib=L)
        assert np.array_equal(yp, y[p])


def pin_slot_relabel(L):
    """Moving adapters to other slots (and remapping ids) leaves y unchanged."""
    x, W, adapters, ids = rand_case(18)
    S = len(adapters)
    q = np.random.default_rng(180).permutation(S)  # adapter in old slot s moves to q[s]
    moved = [None] * S
    for s in range(S):
        moved[q[s]] = adapters[s]
    ids2 = np.where(ids >= 0, q[np.maximum(ids, 0)], -1).astype(np.int32)
    t1 = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    t2 = oracle.SlotTable(moved, W.shape[0], W.shape[1])
    for f in (oracle.forward_rows, oracle.forward_grouped, oracle.forward_merged):
        close(f(x, W, t2, ids2, _lib=L), f(x, W, t1, ids, _lib=L), rel=1e-13)


def pin_padding_ignored_and_true_rank_scale(L):
    """Slot padding beyond the true rank is never read, and the scale uses the true
    rank: fill the padding with garbage and compare with a table of exact width."""
    x, W, adapters, ids = rand_case(19, ranks=(2, 1, 3, 2))
    tight = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    wide = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    R = 6
    wide.R = R
    A = np.full((wide.S, wide.K, R), 7.5)
    B = np.full((wide.S, R, wide.N), -3.25)
    for s, (a, b, _) in enumerate(adapters):
        r = a.shape[1]
        A[s, :, :r] = a
        B[s, :r, :] = b
    wide.A, wide.B = np.ascontiguousarray(A), np.ascontiguousarray(B)
    for f in (oracle.forward_rows, oracle.forward_grouped, oracle.forward_merged):
        close(f(x, W, wide, ids, _lib=L), f(x, W, tight, ids, _lib=L))


def pin_bad_ids(L):
    """Ids outside [-1, S) are counted and treated as base only."""
    x, W, adapters, ids = rand_case(20)
    S = len(adapters)
    bad_ids = ids.copy()
    bad_ids[[1, 5, 9]] = [S, -2, S + 7]
    _, _, _, bad = oracle.segments(bad_ids, S, _lib=L)
    assert bad == 3
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    as_base = bad_ids.copy()
    as_base[[1, 5, 9]] = -1
    for f in (oracle.forward_rows, oracle.forward_grouped, oracle.forward_merged):
        close(f(x, W, table, bad_ids, _lib=L), f(x, W, table, as_base, _lib=L), rel=0)


# --------------------------------------------------------------------------------
# Brute force on tiny inputs
# --------------------------------------------------------------------------------

def pin_segments_brute_force(L):
    """The builder equals Python's stable ``sorted`` of the adapted rows by slot, over
    every id vector of length 5 on {-1, 0, 1, 2} and random longer ones."""
    cases = [np.array(c, np.int32) for c in itertools.product((-1, 0, 1, 2), repeat=5)]
    rng = np.random.default_rng(21)
    cases += [rng.integers(-1, 9, size=int(rng.integers(1, 300))).astype(np.int32)
              for _ in range(60)]
    for ids in cases:
        S = int(max(ids.max() + 1, 1)) + 1
        perm, offs, sslot, bad = oracle.segments(ids, S, _lib=L)
        adapted = [i for i in range(len(ids)) if ids[i] >= 0]
        expect = sorted(adapted, key=lambda i: ids[i])
        assert bad == 0 and perm.tolist() == expect
        used = sorted(set(int(ids[i]) for i in adapted))
        assert sslot.tolist() == used
        counts = [int((ids == s).sum()) for s in used]
        assert offs.tolist() == [0] + list(np.cumsum(counts)) if used else offs.tolist() == [0]


def pin_exact_integers(L):
    """Small-integer inputs make every fp64 sum exact: compare with exact integer
    arithmetic of the definition, row by row."""
    rng = np.random.default_rng(22)
    T, K, N, S = 7, 5, 4, 3
    x = rng.integers(-3, 4, size=(T, K))
    W = rng.integers(-3, 4, size=(K, N))
    ranks = (2, 1, 3)
    adapters = [(rng.integers(-2, 3, size=(K, r)), rng.integers(-2, 3, size=(r, N)),
                 float(2 * r)) for r in ranks]  # alpha = 2 r: scale exactly 2
    ids = np.array([0, -1, 2, 1, 2, 0, -1], np.int32)
    exact = []
    for i in range(T):
        row = [sum(int(x[i, k]) * int(W[k, n]) for k in range(K)) for n in range(N)]
        if ids[i] >= 0:
            A, B, _ = adapters[ids[i]]
            r = A.shape[1]
            v = [sum(int(x[i, k]) * int(A[k, j]) for k in range(K)) for j in range(r)]
            row = [row[n] + 2 * sum(v[j] * int(B[j, n]) for j in range(r)) for n in range(N)]
        exact.append(row)
    table = oracle.SlotTable([(A.astype(float), B.astype(float), a) for A, B, a in adapters], K, N)
    for out in all_evaluators(L, x.astype(float), W.astype(float), table, ids):
        assert np.array_equal(out, np.array(exact, dtype=np.float64))




def pin_row_subset(L):
    """Evaluating a sample of rows gives exactly those rows of the full evaluation."""
    x, W, adapters, ids = rand_case(23, T=33)
    table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
    full = oracle.forward_rows(x, W, table, ids, _lib=L)
    pick = np.array([32, 0, 7, 7, 19], dtype=np.int64)
    assert np.array_equal(oracle.forward_rows(x, W, table, ids, rows=pick, _lib=L), full[pick])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
