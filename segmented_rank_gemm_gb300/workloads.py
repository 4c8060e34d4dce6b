"""Seeded synthetic inputs for the mixed-adapter LoRA layer.

This module only draws tensors and token->slot maps.  It holds none of the layer's
arithmetic, imports neither the CUDA binding nor the oracle, and serves both: the
tests and the benchmark feed the same drawn values to the CUDA path and to the CPU
oracle.

Each recipe follows the workload shapes the pages describe (8B-class projections,
rank 8-64, about a hundred resident adapter slots) and the readings written down in
the design notes: how segment lengths, popularity and base-only rows are drawn.

A ``Workload`` holds:
  x           [T, K]   activations (bf16, or fp32 for the worked example)
  W           [K, N]   shared base weight
  adapters    list of length S: ``None`` (empty slot) or ``(A [K, r], B [r, N], alpha)``
  token_slot  int32 [T], the slot of each row, -1 = base only
  R           slot rank width (the padded width of the slot table)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

BF16 = torch.bfloat16
F32 = torch.float32


@dataclasses.dataclass
class Workload:
    name: str
    x: torch.Tensor
    W: torch.Tensor
    adapters: list
    token_slot: torch.Tensor
    R: int
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.x.shape[0])

    @property
    def K(self) -> int:
        return int(self.W.shape[0])

    @property
    def N(self) -> int:
        return int(self.W.shape[1])

    @property
    def S(self) -> int:
        return len(self.adapters)

    @property
    def dtype(self) -> torch.dtype:
        return self.x.dtype


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(g, shape, std: float, dtype, device="cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


# ---------------------------------------------------------------------------------
# The worked examples printed on the pages
# ---------------------------------------------------------------------------------

def worked_example() -> Workload:
    """6 token rows, K=8, N=5, rank 2, fp32, seed 241 ("Multi-LoRA Serving 与 Adapter
    隔离", grouped-batch experiment).  Draw order as on the page: W[8,5], A_fin[8,2],
    B_fin[2,5], A_code[8,2], B_code[2,5], x[6,8], from torch's CPU generator.
    Slots: finance -> 0 (alpha 4), code -> 1 (alpha 2); base -> -1."""
    torch.manual_seed(241)
    W = torch.randn(8, 5, dtype=F32)
    a_fin, b_fin = torch.randn(8, 2), torch.randn(2, 5)
    a_code, b_code = torch.randn(8, 2), torch.randn(2, 5)
    x = torch.randn(6, 8, dtype=F32)
    names = ["finance", "base", "code", "finance", "code", "base"]
    slot_of = {"finance": 0, "code": 1, "base": -1}
    ids = torch.tensor([slot_of[n] for n in names], dtype=torch.int32)
    return Workload("worked_example", x, W, [(a_fin, b_fin, 4.0), (a_code, b_code, 2.0)],
                    ids, R=2, meta={"row_names": names})


def handbook_toy() -> Workload:
    """The mixed batch of "Serving multiple LoRAs: segmented matrix multiplies and
    adapter scheduling": seed 0, D_in = D_out = 256, rank 16, 8 adapters, scale 2.0
    (alpha = 32 so that alpha / r = 2), request lengths [1,1,37,1,12,1] with adapters
    [3,5,3,0,7,5]; draw order W, A, B, x; every row adapted."""
    torch.manual_seed(0)
    d_in, d_out, r, n_ad = 256, 256, 16, 8
    W = torch.randn(d_in, d_out) / 16
    A = torch.randn(n_ad, d_in, r) / 16
    B = torch.randn(n_ad, r, d_out) / 4
    lengths, owners = [1, 1, 37, 1, 12, 1], [3, 5, 3, 0, 7, 5]
    x = torch.randn(sum(lengths), d_in)
    ids = torch.tensor([a for a, n in zip(owners, lengths) for _ in range(n)], dtype=torch.int32)
    adapters = [(A[i].clone(), B[i].clone(), 2.0 * r) for i in range(n_ad)]
    return Workload("handbook_toy", x, W, adapters, ids, R=r,
                    meta={"lengths": lengths, "owners": owners})


# ---------------------------------------------------------------------------------
# Full-size recipes (8B-class shapes)
# ---------------------------------------------------------------------------------

def decode_bgmv(seed: int = 1002, T: int = 256, K: int = 4096, N: int = 4096, r: int = 16,
                S: int = 128, base_frac: float = 0.1, alpha: float = 32.0,
                dtype=BF16, device="cpu") -> Workload:
    """Decode batch: one token per request; each token independently base-only with
    probability ``base_frac``, else a slot uniform over ``S``; x ~ N(0,1),
    W, A, B ~ N(0, 0.02)."""
    g = _gen(seed, device)
    W = _randn(g, (K, N), 0.02, dtype, device)
    adapters = [(_randn(g, (K, r), 0.02, dtype, device), _randn(g, (r, N), 0.02, dtype, device),
                 alpha) for _ in range(S)]
    x = _randn(g, (T, K), 1.0, dtype, device)
    rng = np.random.default_rng(seed)
    base = rng.random(T) < base_frac
    ids = rng.integers(0, S, size=T)
    ids[base] = -1
    return Workload("decode_bgmv", x, W, adapters, torch.tensor(ids, dtype=torch.int32), R=r,
                    meta={"alpha": alpha, "base_frac": base_frac})


def geometric_lengths(rng: np.random.Generator, n: int, mean: int, total: int) -> np.ndarray:
    """n lengths drawn Geometric(p = 1/mean) on {1, 2, ...}, rescaled to sum to
    ``total``: floor(l * total / sum) clamped to >= 1, the remainder handed out one by
    one to the largest fractional parts first (ties to the lower index)."""
    raw = rng.geometric(1.0 / mean, size=n).astype(np.float64)
    scaled = raw * total / raw.sum()
    base = np.maximum(np.floor(scaled).astype(np.int64), 1)
    rem = total - int(base.sum())
    frac = scaled - np.floor(scaled)
    order = sorted(range(n), key=lambda i: (-frac[i], i))
    i = 0
    while rem > 0:
        base[order[i % n]] += 1
        rem -= 1
        i += 1
    while rem < 0:  # only when clamping to 1 overshot: take from the longest
        j = int(np.argmax(base))
        base[j] -= 1
        rem += 1
    assert int(base.sum()) == total and base.min() >= 1
    return base


def prefill_sgmv(seed: int = 1003, T: int = 8192, n_seg: int = 32, mean_len: int = 256,
                 K: int = 4096, N: int = 14336, ranks=(8, 16, 32, 64), R: int = 64,
                 dtype=BF16, device="cpu") -> Workload:
    """Prefill batch: ``n_seg`` contiguous segments with geometric lengths summing to
    T; segment j is owned by slot sigma(j) (a seeded permutation, so token order is
    not slot order); true ranks uniform over ``ranks``, alpha = 2 r, padded in an
    R-wide slot; weights ~ N(0, 0.02), x ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    lengths = geometric_lengths(rng, n_seg, mean_len, T)
    sigma = rng.permutation(n_seg)
    true_rank = rng.choice(np.asarray(ranks), size=n_seg)
    g = _gen(seed, device)
    W = _randn(g, (K, N), 0.02, dtype, device)
    adapters = []
    for s in range(n_seg):
        r = int(true_rank[s])
        adapters.append((_randn(g, (K, r), 0.02, dtype, device),
                         _randn(g, (r, N), 0.02, dtype, device), 2.0 * r))
    x = _randn(g, (T, K), 1.0, dtype, device)
    ids = np.concatenate([np.full(int(l), int(sigma[j])) for j, l in enumerate(lengths)])
    return Workload("prefill_sgmv", x, W, adapters, torch.tensor(ids, dtype=torch.int32), R=R,
                    meta={"lengths": lengths.tolist(), "sigma": sigma.tolist(),
                          "ranks": true_rank.tolist()})


def zipf_probs(n_ids: int, s: float) -> np.ndarray:
    p = np.arange(1, n_ids + 1, dtype=np.float64) ** (-s)
    return p / p.sum()


def mixed_continuous(seed: int = 1004, n_prefill: int = 8, prefill_len: int = 448,
                     n_decode: int = 512, K: int = 14336, N: int = 4096, r: int = 16,
                     n_ids: int = 1000, S: int = 100, zipf_s: float = 1.1,
                     alpha: float = 32.0, dtype=BF16, device="cpu") -> Workload:
    """Continuous batch: ``n_prefill`` prefill requests of ``prefill_len`` rows plus
    ``n_decode`` one-row decode requests, in a seeded random request order (each
    prefill request contiguous).  Each request draws an adapter id k in 1..n_ids with
    P(k) ~ k^-zipf_s and uses slot (k - 1) mod S.  No base-only rows."""
    rng = np.random.default_rng(seed)
    p = zipf_probs(n_ids, zipf_s)
    n_req = n_prefill + n_decode
    req_ids = rng.choice(np.arange(1, n_ids + 1), size=n_req, p=p)
    req_len = np.array([prefill_len] * n_prefill + [1] * n_decode)
    order = rng.permutation(n_req)
    ids = np.concatenate([np.full(int(req_len[q]), int((req_ids[q] - 1) % S)) for q in order])
    g = _gen(seed, device)
    W = _randn(g, (K, N), 0.02, dtype, device)
    adapters = [(_randn(g, (K, r), 0.02, dtype, device), _randn(g, (r, N), 0.02, dtype, device),
                 alpha) for _ in range(S)]
    T = int(req_len.sum())
    x = _randn(g, (T, K), 1.0, dtype, device)
    return Workload("mixed_continuous", x, W, adapters, torch.tensor(ids, dtype=torch.int32),
                    R=r, meta={"request_order": order.tolist()})


# The 8B-class LoRA stack: 32 layers x 7 projections, rank 16, 100 resident slots.
STACK_PROJECTIONS = (("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024),
                     ("o", 4096, 4096), ("gate", 4096, 14336), ("up", 4096, 14336),
                     ("down", 14336, 4096))


def stack_tokens(seed: int = 1005, T: int = 512, K: int = 4096, S: int = 100,
                 dtype=BF16, device="cpu"):
    """Input rows h0 ~ N(0,1) [T, K] and uniform slot ids over S (no base-only rows)."""
    rng = np.random.default_rng(seed)
    ids = torch.tensor(rng.integers(0, S, size=T), dtype=torch.int32)
    g = _gen(seed, device)
    h0 = _randn(g, (T, K), 1.0, dtype, device)
    return h0, ids


def stack_projection(layer: int, proj: int, seed: int = 1005, S: int = 100, r: int = 16,
                     alpha: float = 32.0, dtype=BF16, device="cpu"):
    """Weights of projection ``proj`` (index into STACK_PROJECTIONS) of ``layer``:
    W ~ N(0, 0.02) [K, N] and S adapters' (A [K, r], B [r, N], alpha), each drawn
    from its own seed so any projection can be regenerated on its own."""
    _, K, N = STACK_PROJECTIONS[proj]
    g = _gen(seed * 1000 + layer * 16 + proj + 1, device)
    W = _randn(g, (K, N), 0.02, dtype, device)
    adapters = [(_randn(g, (K, r), 0.02, dtype, device), _randn(g, (r, N), 0.02, dtype, device),
                 alpha) for _ in range(S)]
    return W, adapters


def stack_input(proj: int, T: int = 512, seed: int = 1005, dtype=BF16, device="cpu"):
    """A fresh N(0,1) input [T, K] for projection ``proj`` of the stack: the per-projection
    parity cases feed every projection an input of its own instead of the previous
    projection's output."""
    _, K, _ = STACK_PROJECTIONS[proj]
    g = _gen(seed * 7919 + proj + 17, device)
    return _randn(g, (T, K), 1.0, dtype, device)


# ---------------------------------------------------------------------------------
# Generic seeded cases for the tests
# ---------------------------------------------------------------------------------

def synthetic(seed: int, T: int, K: int, N: int, S: int, ranks, R: Optional[int] = None,
              dtype=BF16, base_frac: float = 0.1, layout: str = "random",
              empty_slots=(), x_std: float = 1.0, w_std: float = 0.02,
              alpha_per_rank: float = 2.0, device="cpu") -> Workload:
    """A seeded case of any shape.  ``ranks`` is one rank for all slots or a list per
    slot; ``layout`` is ``random`` (ids drawn per row), ``sorted`` (rows already grouped
    by ascending slot) or ``runs`` (random runs of equal ids).  Slots listed in
    ``empty_slots`` hold no adapter."""
    rng = np.random.default_rng(seed)
    ranks = [int(ranks)] * S if np.isscalar(ranks) else [int(v) for v in ranks]
    R = R if R is not None else (max(ranks) if ranks else 1)
    g = _gen(seed, device)
    W = _randn(g, (K, N), w_std, dtype, device)
    adapters = []
    for s in range(S):
        if s in empty_slots:
            adapters.append(None)
            continue
        r = ranks[s]
        adapters.append((_randn(g, (K, r), w_std, dtype, device),
                         _randn(g, (r, N), w_std, dtype, device), alpha_per_rank * r))
    x = _randn(g, (T, K), x_std, dtype, device)
    live = [s for s in range(S) if s not in empty_slots]
    if layout == "runs":
        ids = []
        while len(ids) < T:
            run = int(rng.integers(1, 64))
            sid = -1 if (rng.random() < base_frac or not live) else int(rng.choice(live))
            ids.extend([sid] * run)
        ids = np.asarray(ids[:T])
    else:
        ids = rng.choice(live, size=T) if live else np.full(T, -1)
        ids = np.where(rng.random(T) < base_frac, -1, ids)
        if layout == "sorted":
            ids = np.sort(ids)
    return Workload("synthetic", x, W, adapters, torch.tensor(ids, dtype=torch.int32), R=R,
                    meta={"seed": seed, "layout": layout})
