"""The adapter cache on the GPU, through the C ABI: layers whose slots are filled only by
swap-ins from the cache's host tier, checked against the oracle evaluated on the adapters
by id (not by slot), so every eviction and reload must put the right weights in the right
slot of every layer.

Layers of three kinds share the cache: bf16 (delta mode up to 512 rows, tensor-core expand
with the B expand pool above), a second bf16 shape, and fp32.  Batches alternate between
200 and 600 rows, name at most as many adapters as there are slots, and are chosen so
that most of them swap something in.  The tests run over plain layers (slot s at rows
s R .. s R + R) and over pooled ones (each adapter at its rank rounded up to 8 rows, placed
by the pool's first-fit allocator at every swap-in: ranks 1 .. 16 in this universe move
slots between runs of 8 and 16 rows, so rows are freed and taken again all the time).
"""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32

N_IDS, SLOTS = 9, 4
RANKS = [1, 16, 8, 3, 12, 16, 2, 5, 9]
SHAPES = [(256, 192, BF16), (128, 264, BF16), (72, 40, F32)]  # K, N, dtype
T_MAX = 640


def _universe():
    """Per layer: W and the N_IDS adapters (index = adapter id)."""
    return [workloads.synthetic(900 + i, 1, K, N, S=N_IDS, ranks=RANKS, R=16, dtype=dt,
                                base_frac=0.0)
            for i, (K, N, dt) in enumerate(SHAPES)]


def _build(wls, slots=SLOTS, host=N_IDS, pooled=False):
    from segmented_rank_gemm_gb300.lora import AdapterCache, LoraLayer
    # pooled: room for every slot at rank 16 plus two spare runs (fragmentation)
    pool = 16 * (slots + 2) if pooled else 0
    layers = [LoraLayer(wl.W.cuda(), slots + 2, 16, T_MAX, pool_rows=pool) for wl in wls]
    cache = AdapterCache(layers, slots, host)
    for a in range(N_IDS):
        cache.add(a, [wl.adapters[a][0] for wl in wls], [wl.adapters[a][1] for wl in wls],
                  wls[0].adapters[a][2])
    return layers, cache


def _run_batch(layers, cache, wls, ids, seed, stream):
    """Map, forward every layer on `stream`; returns the outputs and their inputs."""
    slots = cache.map_batch(ids, stream)
    g = torch.Generator().manual_seed(seed)
    outs = []
    with torch.cuda.stream(stream):  # every device buffer of the batch is made on `stream`
        tok = torch.from_numpy(slots.astype(np.int32)).cuda()
        for L, wl in zip(layers, wls):
            x = torch.randn(len(ids), wl.K, generator=g).to(wl.dtype)
            outs.append((x, L(x.cuda(), tok, stream=stream)))
    return slots, outs


def _check(wls, ids, outs, what):
    for wl, (x, y) in zip(wls, outs):
        table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
        ref = oracle.forward_rows(x, wl.W, table, torch.tensor(ids, dtype=torch.int32))
        assert_parity(y, ref, wl.dtype, what="%s K=%d N=%d" % (what, wl.K, wl.N))


@pytest.mark.parametrize("pooled", [False, True], ids=["plain", "pooled"])
def test_swaps_keep_parity_over_a_batch_sequence(pooled):
    from segmented_rank_gemm_gb300.lora import LoraError
    wls = _universe()
    layers, cache = _build(wls, pooled=pooled)
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(11)
    pending = []
    for step in range(10):
        T = 200 if step % 2 == 0 else 600
        names = rng.choice(N_IDS, size=int(rng.integers(1, SLOTS + 1)), replace=False)
        ids = np.where(rng.random(T) < 0.1, -1, rng.choice(names, size=T)).astype(np.int64)
        slots, outs = _run_batch(layers, cache, wls, ids, step, stream)
        for a in set(ids.tolist()) - {-1}:
            assert slots[ids == a][0] == cache.slot_of(a)
        pending.append((ids, outs))
        if step % 3 == 2:  # prefetch an adapter beside this batch, if a slot is free of it
            try:
                cache.prefetch(rng.choice(N_IDS, size=1))
            except LoraError as e:
                assert e.code == -10  # LORA_ECAPACITY: every slot serves the running batch
    torch.cuda.synchronize()
    for step, (ids, outs) in enumerate(pending):
        _check(wls, ids, outs, "step %d" % step)
    for L in layers:
        assert L.status(stream) == 0
    st = cache.stats()
    assert st["misses"] >= 6 and st["gpu_evictions"] >= 3, st
    image = sum(16 * (wl.K + wl.N) * (2 if wl.dtype == BF16 else 4) for wl in wls)
    assert st["bytes_swapped"] >= (st["misses"] + st["prefetches"]) * image
    if pooled:  # the resident adapters hold exactly their ranks rounded up to 8 rows
        want = sum((RANKS[a] + 7) // 8 * 8 for a in range(N_IDS) if cache.slot_of(a) >= 0)
        for L in layers:
            assert L.pool_usage()[0] == want
    cache.close()


@pytest.mark.parametrize("pooled", [False, True], ids=["plain", "pooled"])
def test_one_slot_eviction_under_a_running_batch(pooled):
    """One slot: each batch evicts the previous batch's adapter right after that batch's
    forwards were enqueued (no host synchronisation), so the swap-in must wait for them
    (pooled: the new adapter reuses rows the running batch reads)."""
    wls = _universe()
    layers, cache = _build(wls, slots=1, host=N_IDS, pooled=pooled)
    stream = torch.cuda.Stream()
    runs = []
    for step, a in enumerate([0, 5, 1, 5, 8, 2]):
        ids = np.full(200 if step % 2 else 600, a, np.int64)
        ids[::7] = -1
        runs.append((ids, _run_batch(layers, cache, wls, ids, 100 + step, stream)[1]))
    torch.cuda.synchronize()
    for step, (ids, outs) in enumerate(runs):
        _check(wls, ids, outs, "one-slot step %d" % step)
    assert cache.stats()["gpu_evictions"] == 5
    cache.close()


@pytest.mark.parametrize("pooled", [False, True], ids=["plain", "pooled"])
def test_replace_and_remove(pooled):
    wls = _universe()
    layers, cache = _build(wls, pooled=pooled)
    stream = torch.cuda.Stream()
    ids = np.array([3, 4, -1, 3, 4] * 40, np.int64)
    _run_batch(layers, cache, wls, ids, 1, stream)
    # adapter 3 gets new weights under the same id (in place) while that batch may run
    new3 = [workloads.synthetic(950 + i, 1, wl.K, wl.N, S=1, ranks=[7], R=16, dtype=wl.dtype)
            .adapters[0] for i, wl in enumerate(wls)]
    cache.add(3, [a[0] for a in new3], [a[1] for a in new3], new3[0][2])
    for wl, a in zip(wls, new3):
        wl.adapters[3] = a
    _, outs = _run_batch(layers, cache, wls, ids, 2, stream)
    torch.cuda.synchronize()
    _check(wls, ids, outs, "after replacing adapter 3")
    # removing adapter 4 empties its slot: a forged batch still naming that slot computes
    # base only and raises the layers' id flag
    slot4 = cache.slot_of(4)
    cache.remove(4)
    cache.map_batch(np.array([3], np.int64), stream)  # the next batch point empties it
    base = torch.full((64,), -1, dtype=torch.int32)
    with torch.cuda.stream(stream):
        forged = torch.full((64,), slot4, dtype=torch.int32, device="cuda")
        for L, wl in zip(layers, wls):
            x = torch.randn(64, wl.K, generator=torch.Generator().manual_seed(5)).to(wl.dtype)
            y = L(x.cuda(), forged, stream=stream)
            torch.cuda.synchronize()
            table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
            ref = oracle.forward_rows(x, wl.W, table, base)
            assert_parity(y, ref, wl.dtype, what="removed slot, base only")
            assert L.status(stream) == -4  # LORA_EID
    with pytest.raises(Exception):
        cache.map_batch(np.array([4], np.int64), stream)
    cache.close()


def test_swap_in_through_many_layers_and_capacity_errors():
    """Twenty layers in one image (one copy + one scatter launch per swap-in), and the
    batch-level capacity error of the pages (more adapters than slots)."""
    from segmented_rank_gemm_gb300.lora import AdapterCache, LoraError, LoraLayer
    wl = workloads.synthetic(990, 1, 128, 136, S=6, ranks=[4, 8, 16, 2, 9, 16], R=16,
                             base_frac=0.0)
    layers = [LoraLayer(wl.W.cuda(), 3, 16, 256) for _ in range(20)]
    cache = AdapterCache(layers, 3, 6)
    for a in range(6):
        A, B, alpha = wl.adapters[a]
        cache.add(a, [A] * 20, [B] * 20, alpha)
    with pytest.raises(LoraError) as e:
        cache.map_batch(np.array([0, 1, 2, 3], np.int64))
    assert e.value.code == -10  # LORA_ECAPACITY
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(3)
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    for step in range(6):
        names = rng.choice(6, size=3, replace=False)
        ids = rng.choice(names, size=256).astype(np.int64)
        slots = cache.map_batch(ids, stream)
        x = torch.randn(256, wl.K, dtype=BF16)
        with torch.cuda.stream(stream):
            tok = torch.from_numpy(slots.astype(np.int32)).cuda()
            ys = [L(x.cuda(), tok, stream=stream) for L in layers]
        torch.cuda.synchronize()
        ref = oracle.forward_rows(x, wl.W, table, torch.tensor(ids, dtype=torch.int32))
        for y in ys[::7]:
            assert_parity(y, ref, BF16, what="20-layer image, step %d" % step)
    cache.close()


@pytest.mark.parametrize("pooled", [False, True], ids=["plain", "pooled"])
def test_composed_adapters_through_the_cache(pooled):
    """Compositions held under their own ids beside plain adapters: packed from the members'
    host blocks (so removing a member later leaves them intact), swapped in like any
    adapter, rows naming them add their members' weighted deltas."""
    wls = _universe()
    layers, cache = _build(wls, host=N_IDS + 4, pooled=pooled)
    compositions = {20: ([0, 3, 7], [0.5, -1.0, 2.0]), 21: ([2, 6], [1.0, 0.25]),
                    22: ([2, 2], [0.5, 0.5])}
    for cid, (members, weights) in compositions.items():
        cache.add_composed(cid, members, weights)
    cache.remove(7)  # the composition 20 keeps its own copy
    per_layer = []
    for wl in wls:
        comps = {a: [(A, B, al, 1.0)] for a, (A, B, al) in enumerate(wl.adapters)}
        for cid, (members, weights) in compositions.items():
            comps[cid] = [(*wl.adapters[m], w) for m, w in zip(members, weights)]
        per_layer.append(comps)
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(21)
    runs = []
    for step, names in enumerate([[20, 1], [21, 22, 20], [0, 21, 5, 22], [20, 21]]):
        T = 200 if step % 2 == 0 else 600
        ids = np.where(rng.random(T) < 0.1, -1, rng.choice(names, size=T)).astype(np.int64)
        runs.append((ids, _run_batch(layers, cache, wls, ids, 300 + step, stream)[1]))
    torch.cuda.synchronize()
    for step, (ids, outs) in enumerate(runs):
        for wl, comps, (x, y) in zip(wls, per_layer, outs):
            order = sorted(comps)
            index = {a: i for i, a in enumerate(order)}
            slot_ids = torch.tensor([index[int(a)] if a >= 0 else -1 for a in ids],
                                    dtype=torch.int32)
            ref = oracle.forward_composed(x, wl.W, [comps[a] for a in order], slot_ids)
            assert_parity(y, ref, wl.dtype, what="composed ids, step %d K=%d" % (step, wl.K))
    for L in layers:
        assert L.status(stream) == 0
    cache.close()


def test_pooled_rows_exhausted_leaves_the_slot_empty():
    """A pool too small for the adapter a batch needs: map_batch fails with LORA_ENOMEM, the
    slot is left empty in every layer, and the cache keeps serving what fits."""
    from segmented_rank_gemm_gb300.lora import AdapterCache, LoraError, LoraLayer
    wls = _universe()[:2]
    # 24 rows: adapter 1 (rank 16: 16 rows) and adapter 0 (rank 1: 8 rows) fit together;
    # adapter 5 (rank 16) then needs 16 free rows while 8 are left
    layers = [LoraLayer(wl.W.cuda(), 4, 16, T_MAX, pool_rows=24) for wl in wls]
    cache = AdapterCache(layers, 3, N_IDS)
    for a in range(N_IDS):
        cache.add(a, [wl.adapters[a][0] for wl in wls], [wl.adapters[a][1] for wl in wls],
                  wls[0].adapters[a][2])
    stream = torch.cuda.Stream()
    ids = np.array([1, 0, -1, 1] * 50, np.int64)
    _, outs = _run_batch(layers, cache, wls, ids, 7, stream)
    torch.cuda.synchronize()
    _check(wls, ids, outs, "pool of 24 rows, adapters 1 and 0")
    with pytest.raises(LoraError) as e:
        cache.map_batch(np.array([1, 0, 5], np.int64), stream)
    assert e.value.code == -6  # LORA_ENOMEM
    assert cache.slot_of(5) == -1 and cache.slot_of(1) >= 0 and cache.slot_of(0) >= 0
    for L in layers:
        assert L.pool_usage()[0] == 24
    # the adapters that fit are still served correctly
    ids = np.array([0, 1, 1, -1] * 40, np.int64)
    _, outs = _run_batch(layers, cache, wls, ids, 8, stream)
    torch.cuda.synchronize()
    _check(wls, ids, outs, "after a refused swap-in")
    for L in layers:
        assert L.status(stream) == 0
    cache.close()
