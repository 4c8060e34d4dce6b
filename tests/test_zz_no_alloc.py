"""The allocation-free segment builder (lora_build_segments_static) against the layer's
own set_batch_segments + lora_get_segments, through the C ABI.

lora_build_segments_static is for callers that may not allocate device memory (engines
that own all memory through their own pool, latency-critical paths that cannot afford
cudaMalloc's synchronisation): its scratch is a static device array shared by all calls.
Two calls in a row with different batches check that nothing of the first call's leftover
state (scratch contents, error flags) leaks into the second.  Segment layouts are integer
results, so the comparison is bit-exact.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _reference(ids, S, loaded_slots):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    T = len(ids)
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    layer = LoraLayer(W, S, 2, max(T, 1))
    A = torch.zeros(64, 1, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    for s in loaded_slots:
        layer.load(s, A, B, 1.0)
    layer.set_batch(torch.from_numpy(np.asarray(ids, np.int32)).cuda())
    perm, offs, sslot = layer.segments()
    status = layer.status()
    layer.close()
    return perm, offs, sslot, status


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


def test_static_builder_matches_layer_on_two_calls_in_a_row():
    rng = np.random.default_rng(2024)
    S = 96
    # call 1: a decode-like batch with ids outside the table and one empty slot
    ids1 = rng.integers(-1, S, size=777)
    ids1[[3, 50, 400]] = [S + 5, -3, S]
    loaded1 = np.ones(S, np.int32)
    loaded1[7] = 0
    # call 2: a prefill-like batch of long runs, every slot loaded, fewer rows
    ids2 = np.repeat(rng.integers(-1, S, size=25), rng.integers(1, 40, size=25))[:500]

    for ids, loaded in ((ids1, loaded1), (ids2, None)):
        ref_perm, ref_offs, ref_slot, ref_status = _reference(
            ids, S, [s for s in range(S) if loaded is None or loaded[s]])
        perm, offs, sslot, flags = _static(ids, S, loaded)
        assert np.array_equal(perm, ref_perm)
        assert np.array_equal(offs, ref_offs)
        assert np.array_equal(sslot, ref_slot)
        assert (flags != 0) == (ref_status != 0)  # bad ids flagged only in the first batch


def test_static_builder_rejects_oversize():
    from segmented_rank_gemm_gb300.lora import LoraError, lora_build_segments_static
    big = torch.zeros(16385, dtype=torch.int32, device="cuda")
    out = torch.zeros(16385, dtype=torch.int32, device="cuda")
    small = torch.zeros(2048, dtype=torch.int32, device="cuda")
    with pytest.raises(LoraError):
        lora_build_segments_static(big, 16385, 8, None, out, small, small, small)
    with pytest.raises(LoraError):
        lora_build_segments_static(small, 16, 1025, None, out, small, small, small)
