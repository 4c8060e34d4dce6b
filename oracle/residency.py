"""Reference model of adapter residency: which adapters sit in which GPU slots, and which
leave the host tier, as a sequence of batches arrives.

TEST INFRASTRUCTURE (part of the oracle package).  Plain Python lists and dicts, one step
at a time, written from the pages' description; it shares no code with the library's cache
and never imports it.

The policy, by page:
- "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM), Step 3:
  * a batch naming more distinct adapters than GPU slots is rejected;
  * an adapter missing from the CPU cache is loaded into it, after a validity check and
    before anything is evicted; a full CPU cache removes its oldest adapter;
  * activation puts an adapter into the first free slot; with every slot taken, the
    least recently used active adapter is deactivated first;
  * an adapter already loaded is only touched (its recency refreshed).
- "Multi-LoRA Serving: Architecture for Thousands of Adapters", section "Trade-offs,
  Gotchas, and What Goes Wrong": eviction is LRU, and traffic cycling over more adapters
  than fit thrashes the cache.
- "LoRAX, in depth", section "Adapter exchange scheduling": adapters with queued work are
  prefetched.

Readings where the pages leave a step open (the library follows the same ones):
- a batch's adapters are handled in the order of their first row, and each is touched when
  handled, so a batch's first-named adapter is the least recent of its adapters afterwards;
- a slot is never taken from an adapter the same batch (or prefetch list) names;
- the host tier holds every adapter that may be resident; dropping the oldest host adapter
  also frees its GPU slot, whether or not it was resident;
- adding an id already held replaces its weights and frees its slot;
- the adapters of the last mapped batch may still be computing ("Multi-LoRA Serving 与
  Adapter 隔离", failure modes: never evict an adapter under an in-flight kernel): a
  prefetch does not take their slots, and a slot whose adapter leaves while that batch
  may run stays blocked until the next batch begins.
"""
from __future__ import annotations


class ResidencyError(Exception):
    """The request is refused; ``kind`` is 'unknown', 'capacity' or 'invalid'."""

    def __init__(self, kind: str):
        super().__init__(kind)
        self.kind = kind


BLOCKED = "blocked"  # a slot whose adapter left while the last batch may still run


class ResidencyModel:
    def __init__(self, num_slots: int, host_capacity: int):
        assert num_slots >= 1 and host_capacity >= num_slots
        self.num_slots = num_slots
        self.host_capacity = host_capacity
        self.slots = [None] * num_slots  # adapter id per GPU slot, None, or BLOCKED
        self.host = []                   # adapter ids in the host tier
        self.recency = []                # every held adapter id, least recent first
        self.last_slots = []             # slots of the last mapped batch
        self.last_names = []             # its adapters
        self.stats = dict(hits=0, misses=0, prefetches=0, gpu_evictions=0, host_evictions=0)

    # -- helpers ------------------------------------------------------------------------
    def _touch(self, a):
        if a in self.recency:
            self.recency.remove(a)
        self.recency.append(a)

    def slot_of(self, a) -> int:
        return self.slots.index(a) if a in self.slots else -1

    def _free_slot_of(self, a):
        if a in self.slots:
            s = self.slots.index(a)
            self.slots[s] = BLOCKED if s in self.last_slots else None

    # -- host tier ----------------------------------------------------------------------
    def add(self, a, valid: bool = True):
        """Load adapter ``a`` into the host tier (``valid=False``: it fails its check)."""
        if not valid:
            raise ResidencyError("invalid")  # checked before anything is evicted
        if a in self.host:                   # in-place replacement
            self._free_slot_of(a)
            self._touch(a)
            return
        if len(self.host) == self.host_capacity:
            oldest = next(b for b in self.recency if b in self.host)
            self.remove(oldest)
            self.stats["host_evictions"] += 1
        self.host.append(a)
        self._touch(a)

    def add_composed(self, a, members):
        """A composition of adapters in the host tier, held under its own id ``a``; room is
        never made by dropping a member."""
        if a < 0 or a in members:
            raise ResidencyError("invalid")
        if any(m not in self.host for m in members):
            raise ResidencyError("unknown")
        if a in self.host:
            self._free_slot_of(a)
            self._touch(a)
            return
        if len(self.host) == self.host_capacity:
            cands = [b for b in self.recency if b in self.host and b not in members]
            if not cands:
                raise ResidencyError("capacity")
            self.remove(cands[0])
            self.stats["host_evictions"] += 1
        self.host.append(a)
        self._touch(a)

    def remove(self, a):
        if a not in self.host:
            raise ResidencyError("unknown")
        self._free_slot_of(a)
        self.host.remove(a)
        self.recency.remove(a)

    # -- GPU tier -----------------------------------------------------------------------
    def _make_resident(self, names, pinned, batch: bool):
        for a in names:
            if a in self.slots:
                if batch:
                    self.stats["hits"] += 1
                self._touch(a)
                continue
            if None in self.slots:
                s = self.slots.index(None)       # the first free slot
            else:
                candidates = [b for b in self.recency if b in self.slots and b not in pinned]
                victim = candidates[0]           # least recently used, not pinned now
                s = self.slots.index(victim)
                self.stats["gpu_evictions"] += 1
            self.slots[s] = a
            self.stats["misses" if batch else "prefetches"] += 1
            self._touch(a)

    def map_batch(self, token_adapter):
        """Row adapter ids (-1 = base only) -> row slots (-1 for base rows)."""
        names = []
        for a in token_adapter:
            if a == -1:
                continue
            if a < -1:
                raise ResidencyError("invalid")
            if a not in self.host:
                raise ResidencyError("unknown")
            if a not in names:
                names.append(a)
        if len(names) > self.num_slots:
            raise ResidencyError("capacity")
        # the previous batch is over: its blocked slots become free
        self.slots = [None if v == BLOCKED else v for v in self.slots]
        self._make_resident(names, names, batch=True)
        self.last_names = list(names)
        self.last_slots = [self.slot_of(a) for a in names]
        return [-1 if a == -1 else self.slot_of(a) for a in token_adapter]

    def prefetch(self, ids):
        names = []
        for a in ids:
            if a < 0:
                raise ResidencyError("invalid")
            if a not in self.host:
                raise ResidencyError("unknown")
            if a not in names:
                names.append(a)
        pinned = names + [a for a in self.last_names if a not in names]
        missing = sum(a not in self.slots for a in names)
        takeable = sum(v is None or (v != BLOCKED and v not in pinned) for v in self.slots)
        if missing > takeable:
            raise ResidencyError("capacity")
        self._make_resident(names, pinned, batch=False)

    def resident(self) -> int:
        return sum(s is not None and s != BLOCKED for s in self.slots)
