"""Adapter residency without a GPU.

1. The reference model (oracle/residency.py) against what fixes its behaviour from outside:
   the textbook LRU fault count of a classic reference string, the LRU stack property
   (a reference hits exactly when fewer than S other adapters were used since its previous
   use), thrashing of a cyclic sweep over S + 1 adapters, capacity and load-before-evict
   rules of vLLM's Step 3, and the in-flight rule (a prefetch or removal never rewrites a
   slot the last batch may still read).  Mistaken copies of the model (MRU victim, last
   free slot, no touch on a hit) fail these pins.
2. The library's cache in its books-only form (no layers, no device) against the model, on
   long random sequences of adds, removes, batches and prefetches: identical slots, errors
   and counters at every step.
"""
import numpy as np
import pytest

from oracle.residency import ResidencyError, ResidencyModel

# "Operating System Concepts" (Silberschatz, Galvin, Gagne), the page-replacement reference
# string: with 3 frames, LRU replacement takes 12 page faults.
TEXTBOOK_STRING = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]
TEXTBOOK_LRU_FAULTS = 12


def run_single(model_cls, seq, S):
    m = model_cls(S, max(S, len(set(seq))))
    for a in sorted(set(seq)):
        m.add(a)
    hits = []
    for a in seq:
        before = m.stats["hits"]
        m.map_batch([a])
        hits.append(m.stats["hits"] > before)
    return m, hits


def stack_distance_hits(seq, S):
    """Hit iff fewer than S distinct other adapters were used since the previous use."""
    out = []
    for i, a in enumerate(seq):
        prev = [j for j in range(i) if seq[j] == a]
        out.append(bool(prev) and len(set(seq[prev[-1] + 1:i])) < S)
    return out


def pins(model_cls):
    """Every pin of the model; raises AssertionError on the first that fails."""
    m, _ = run_single(model_cls, TEXTBOOK_STRING, 3)
    assert m.stats["misses"] == TEXTBOOK_LRU_FAULTS
    rng = np.random.default_rng(5)
    for S in (1, 2, 4):
        seq = [int(v) for v in rng.integers(0, 7, size=60)]
        assert run_single(model_cls, seq, S)[1] == stack_distance_hits(seq, S)
    # a cyclic sweep over S + 1 adapters misses every time
    S = 4
    m, hits = run_single(model_cls, list(range(S + 1)) * 5, S)
    assert not any(hits)
    # first free slots, in the order of first appearance
    m = model_cls(4, 8)
    for a in (10, 11, 12):
        m.add(a)
    assert m.map_batch([12, -1, 10, 12, 11]) == [0, -1, 1, 0, 2]
    # a batch never evicts an adapter it names; more names than slots is refused
    m = model_cls(2, 4)
    for a in (1, 2, 3):
        m.add(a)
    m.map_batch([1])
    m.map_batch([2])
    assert m.map_batch([2, 3]) == [1, 0]  # 1 is the LRU resident adapter not named
    with pytest.raises(ResidencyError):
        m.map_batch([1, 2, 3])
    # load before evict: a refused add leaves a full host tier alone
    m = model_cls(1, 2)
    m.add(1)
    m.add(2)
    with pytest.raises(ResidencyError):
        m.add(3, valid=False)
    assert m.host == [1, 2] and m.stats["host_evictions"] == 0
    # a full host tier drops its oldest adapter, and that adapter's slot with it
    m.map_batch([1])
    m.map_batch([2])
    m.add(3)
    assert 1 not in m.host and m.slot_of(2) == 0 and m.stats["host_evictions"] == 1
    # a prefetch leaves the last batch's adapters alone, and a slot emptied under that
    # batch stays blocked until the next batch begins
    m = model_cls(3, 6)
    for a in range(5):
        m.add(a)
    m.map_batch([0, 1, 2])
    with pytest.raises(ResidencyError):
        m.prefetch([3])  # every slot is in flight
    m.remove(1)
    with pytest.raises(ResidencyError):
        m.prefetch([3])  # a blocked slot is not free
    assert m.map_batch([3]) == [1]  # the next batch frees it: the lowest free slot
    m.prefetch([4])  # takes the LRU of {0, 2}, both out of flight now
    assert m.slot_of(4) == 0 and m.slot_of(3) == 1
    return True


def test_model_pins():
    assert pins(ResidencyModel)


class _MruVictim(ResidencyModel):
    def _make_resident(self, names, pinned, batch):
        for a in names:
            if a in self.slots:
                self.stats["hits"] += batch
                self._touch(a)
                continue
            if None in self.slots:
                s = self.slots.index(None)
            else:
                cand = [b for b in self.recency if b in self.slots and b not in pinned]
                s = self.slots.index(cand[-1])  # mistake: most recently used
            self.slots[s] = a
            self.stats["misses"] += batch
            self._touch(a)


class _LastFreeSlot(ResidencyModel):
    def _make_resident(self, names, pinned, batch):
        for a in names:
            if a in self.slots:
                self.stats["hits"] += batch
                self._touch(a)
                continue
            if None in self.slots:
                s = len(self.slots) - 1 - self.slots[::-1].index(None)  # mistake
            else:
                cand = [b for b in self.recency if b in self.slots and b not in pinned]
                s = self.slots.index(cand[0])
            self.slots[s] = a
            self.stats["misses"] += batch
            self._touch(a)


class _NoTouchOnHit(ResidencyModel):
    def _make_resident(self, names, pinned, batch):
        for a in names:
            if a in self.slots:
                self.stats["hits"] += batch  # mistake: recency not refreshed
                continue
            if None in self.slots:
                s = self.slots.index(None)
            else:
                cand = [b for b in self.recency if b in self.slots and b not in pinned]
                s = self.slots.index(cand[0])
            self.slots[s] = a
            self.stats["misses"] += batch
            self._touch(a)


@pytest.mark.parametrize("mutant", [_MruVictim, _LastFreeSlot, _NoTouchOnHit])
def test_model_pins_catch_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        pins(mutant)


# ---------------------------------------------------------------------------------------
# the library's books against the model
# ---------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def lib():
    from segmented_rank_gemm_gb300 import build
    build.build()
    from segmented_rank_gemm_gb300 import lora
    return lora


KIND = {"unknown": -9, "capacity": -10, "invalid": -1}


def _lib_call(lib, fn, *args):
    try:
        return fn(*args), 0
    except lib.LoraError as e:
        return None, e.code


def _model_call(fn, *args):
    try:
        return fn(*args), 0
    except ResidencyError as e:
        return None, KIND[e.kind]


@pytest.mark.parametrize("seed,S,H,n_ids", [(1, 4, 6, 10), (2, 8, 8, 20), (3, 1, 3, 5),
                                            (4, 16, 40, 60)])
def test_library_books_match_model(lib, seed, S, H, n_ids):
    rng = np.random.default_rng(seed)
    cache = lib.lora_cache_create([], S, H)
    model = ResidencyModel(S, H)
    try:
        for step in range(600):
            op = rng.choice(["add", "add_bad", "compose", "remove", "batch", "prefetch"],
                            p=[0.18, 0.03, 0.04, 0.07, 0.53, 0.15])
            if op == "add":
                a = int(rng.integers(0, n_ids))
                _, rc = _lib_call(lib, lib.lora_cache_add, cache, a, 4, 8.0)
                _, rm = _model_call(model.add, a)
            elif op == "add_bad":  # rank 0 is refused before anything changes
                a = int(rng.integers(0, n_ids))
                _, rc = _lib_call(lib, lib.lora_cache_add, cache, a, 0, 8.0)
                _, rm = _model_call(model.add, a, False)
                rc = -1 if rc == -3 else rc  # the library says which check failed
            elif op == "compose":  # a composition of 1..3 ids (some maybe absent)
                a = int(rng.integers(0, n_ids))
                members = [int(v) for v in rng.choice(n_ids, size=int(rng.integers(1, 4)))]
                _, rc = _lib_call(lib, lib.lora_cache_add_composed, cache, a, members,
                                  [0.5] * len(members))
                _, rm = _model_call(model.add_composed, a, members)
            elif op == "remove":
                a = int(rng.integers(0, n_ids))
                _, rc = _lib_call(lib, lib.lora_cache_remove, cache, a)
                _, rm = _model_call(model.remove, a)
            elif op == "batch":
                T = int(rng.integers(0, 3 * S + 2))
                k = int(rng.integers(1, S + 2))  # sometimes more names than slots
                names = rng.choice(n_ids, size=min(k, n_ids), replace=False)
                ids = np.where(rng.random(T) < 0.15, -1, rng.choice(names, size=T))
                got, rc = _lib_call(lib, lib.lora_cache_map_batch, cache, ids)
                want, rm = _model_call(model.map_batch, [int(v) for v in ids])
                if rc == 0 and rm == 0:
                    assert list(got) == want, (step, ids)
            else:
                ids = rng.integers(0, n_ids, size=int(rng.integers(0, S + 2)))
                _, rc = _lib_call(lib, lib.lora_cache_prefetch, cache, ids)
                _, rm = _model_call(model.prefetch, [int(v) for v in ids])
            assert rc == rm, (step, op, rc, rm)
            st = lib.lora_cache_get_stats(cache)
            for k in model.stats:
                assert st[k] == model.stats[k], (step, k)
            assert st["resident"] == model.resident()
            assert st["registered"] == len(model.host)
            for a in range(n_ids):
                assert lib.lora_cache_slot_of(cache, a) == model.slot_of(a), (step, a)
    finally:
        lib.lora_cache_destroy(cache)


def test_library_rejects_bad_arguments(lib):
    import ctypes
    L = lib.library()
    h = ctypes.c_void_p()
    assert L.lora_cache_create(ctypes.byref(h), None, 0, 0, 4) == lib.LORA_EINVAL
    assert L.lora_cache_create(ctypes.byref(h), None, 0, 4, 3) == lib.LORA_EINVAL  # host < slots
    assert L.lora_cache_create(ctypes.byref(h), None, 1, 4, 4) == lib.LORA_EINVAL  # null layers
    assert L.lora_cache_create(None, None, 0, 4, 4) == lib.LORA_EINVAL
    cache = lib.lora_cache_create([], 2, 2)
    try:
        with pytest.raises(lib.LoraError) as e:
            lib.lora_cache_add(cache, -5, 4, 1.0)
        assert e.value.code == lib.LORA_EINVAL
        with pytest.raises(lib.LoraError) as e:
            lib.lora_cache_map_batch(cache, np.array([3]))
        assert e.value.code == lib.LORA_ENOENT
        lib.lora_cache_add(cache, 3, 4, 1.0)
        with pytest.raises(lib.LoraError) as e:
            lib.lora_cache_map_batch(cache, np.array([3, -2]))
        assert e.value.code == lib.LORA_EINVAL
        assert list(lib.lora_cache_map_batch(cache, np.array([-1, 3, 3]))) == [-1, 0, 0]
        assert lib.lora_cache_stream(cache) == 0  # books only: no device stream
        lib.lora_cache_sync(cache)
    finally:
        lib.lora_cache_destroy(cache)
    lib.lora_cache_destroy(None)
