"""The allocation-free segment builder (lora_build_segments_static) against the oracle's
reference builder, through the C ABI.

lora_build_segments_static is for callers that may not allocate device memory (engines
that own all memory through their own pool, latency-critical paths that cannot afford
cudaMalloc's synchronisation): its scratch is a static device array shared by all calls.
Segment layouts are integer results with exactly one right answer (ascending slot, original
row order within a slot, base-only and bad rows excluded, empty slots omitted), so perm,
seg_offsets and seg_slot are compared bit for bit with ``oracle.segments``.  Rows naming a
slot that holds no adapter are base only by the layer's definition: the oracle receives them
as -1.  Calls run back to back on the same static array, so nothing of one call's leftover
state (scratch contents, error flags) may leak into the next; the sizes reach the array's
limits (16384 rows, 1024 slots), where the builder's walkers re-read the checked slots from
the scratch and its shared memory exceeds 48 KB.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _static(ids, S, loaded_flags):
    from segmented_rank_gemm_gb300.lora import lora_build_segments_static
    T = len(ids)
    tok = torch.from_numpy(np.asarray(ids, np.int32)).cuda()
    loaded = None if loaded_flags is None else torch.from_numpy(
        np.asarray(loaded_flags, np.int32)).cuda()
    perm = torch.full((max(T, 1),), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((S + 1,), -7, dtype=torch.int32, device="cuda")
    sslot = torch.full((S,), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    lora_build_segments_static(tok, T, S, loaded, perm, offs, sslot, counts)
    torch.cuda.synchronize()
    n_seg, n_ad, flags = counts.cpu().tolist()
    return perm.cpu().numpy()[:n_ad], offs.cpu().numpy()[:n_seg + 1], sslot.cpu().numpy()[:n_seg], flags


def _expected(ids, S, loaded_flags):
    """The oracle's builder on the ids with empty-slot rows made base only; also whether a
    device flag must be raised (an id outside [-1, S) or naming an empty slot)."""
    ids = np.asarray(ids, np.int64)
    in_range = (ids >= 0) & (ids < S)
    empty = np.zeros(len(ids), bool)
    if loaded_flags is not None:
        lf = np.asarray(loaded_flags)
        empty[in_range] = lf[ids[in_range]] == 0
    eff = np.where(empty, -1, ids).astype(np.int32)
    perm, offs, sslot, n_bad = oracle.segments(eff, S)
    return perm, offs, sslot, bool(n_bad > 0 or empty.any())


def _skewed(rng, T, S):
    """Run lengths skewed towards a few hot slots: one slot owns ~40% of the rows in long
    runs, the rest is Zipf-like over all slots in short runs, with base-only runs between."""
    ids = []
    hot = int(rng.integers(0, S))
    p = np.arange(1, S + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    while len(ids) < T:
        u = rng.random()
        if u < 0.4:
            ids.extend([hot] * int(rng.integers(64, 1024)))
        elif u < 0.5:
            ids.extend([-1] * int(rng.integers(1, 64)))
        else:
            ids.extend([int(rng.choice(S, p=p))] * int(rng.integers(1, 16)))
    return np.asarray(ids[:T])


def _check(ids, S, loaded):
    perm, offs, sslot, flags = _static(ids, S, loaded)
    rp, ro, rs, must_flag = _expected(ids, S, loaded)
    assert np.array_equal(perm, rp)
    assert np.array_equal(offs, ro)
    assert np.array_equal(sslot, rs)
    assert (flags != 0) == must_flag


def test_static_builder_matches_oracle_on_calls_in_a_row():
    rng = np.random.default_rng(2024)
    S = 96
    # call 1: a decode-like batch with ids outside the table and one empty slot
    ids1 = rng.integers(-1, S, size=777)
    ids1[[3, 50, 400]] = [S + 5, -3, S]
    loaded1 = np.ones(S, np.int32)
    loaded1[7] = 0
    # call 2: a prefill-like batch of long runs, every slot loaded, fewer rows
    ids2 = np.repeat(rng.integers(-1, S, size=25), rng.integers(1, 40, size=25))[:500]
    # calls 3 and 4: the limits of the static array, skewed run lengths; call 4 has fewer
    # rows and slots than call 3, so stale scratch of call 3 would show
    ids3 = _skewed(rng, 16384, 1024)
    loaded3 = np.ones(1024, np.int32)
    loaded3[rng.choice(1024, 40, replace=False)] = 0
    ids4 = _skewed(rng, 9001, 700)
    for ids, S_i, loaded in ((ids1, S, loaded1), (ids2, S, None), (ids3, 1024, loaded3),
                             (ids4, 700, None)):
        _check(ids, S_i, loaded)


def test_static_builder_empty_and_single_row():
    _check(np.zeros(0, np.int64), 4, None)
    _check(np.array([-1]), 1, None)
    _check(np.array([0]), 1, None)


def test_static_builder_rejects_oversize():
    from segmented_rank_gemm_gb300.lora import LoraError, lora_build_segments_static
    big = torch.zeros(16385, dtype=torch.int32, device="cuda")
    out = torch.zeros(16385, dtype=torch.int32, device="cuda")
    small = torch.zeros(2048, dtype=torch.int32, device="cuda")
    with pytest.raises(LoraError):
        lora_build_segments_static(big, 16385, 8, None, out, small, small, small)
    with pytest.raises(LoraError):
        lora_build_segments_static(small, 16, 1025, None, out, small, small, small)


def test_static_builder_rejects_undersized_buffers():
    from segmented_rank_gemm_gb300.lora import LoraError, lora_build_segments_static
    tok = torch.zeros(100, dtype=torch.int32, device="cuda")
    ok = torch.zeros(100, dtype=torch.int32, device="cuda")
    short = torch.zeros(50, dtype=torch.int32, device="cuda")
    with pytest.raises(LoraError):  # perm shorter than T
        lora_build_segments_static(tok, 100, 8, None, short, ok, ok, ok)
    with pytest.raises(LoraError):  # seg_offsets shorter than S + 1
        lora_build_segments_static(tok, 100, 50, None, ok, short, ok, ok)
    with pytest.raises(LoraError):  # wrong dtype
        lora_build_segments_static(tok, 100, 8, None, ok.long(), ok, ok, ok)
