"""ctypes binding of the layer's C ABI (``include/lora_layer.h``) and of the adapter cache
over it (``include/lora_residency.h``).

The functions below carry the C names and only marshal arguments: torch tensors become
raw pointers, torch streams become ``cudaStream_t`` handles, and a negative status
becomes a ``LoraError``.  All computation happens in ``liblora_layer.so``; if the library
has not been built this module raises on import (there is no CPU fallback).

``LoraLayer`` is a small owner object over the same calls (create on construction,
destroy on ``close``/garbage collection).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import library_path

LIB_PATH = library_path()  # the release library, or the debug flavour (LORA_LAYER_LIBRARY=debug)

LORA_F32, LORA_BF16 = 0, 1
STATUS = {0: "LORA_OK", -1: "LORA_EINVAL", -2: "LORA_ESLOT", -3: "LORA_ERANK", -4: "LORA_EID",
          -5: "LORA_ECUDA", -6: "LORA_ENOMEM", -7: "LORA_ESTATE", -8: "LORA_ETIMEOUT",
          -9: "LORA_ENOENT", -10: "LORA_ECAPACITY", -11: "LORA_EBOUNDS"}
LORA_OK, LORA_EINVAL, LORA_ESLOT, LORA_ERANK, LORA_EID = 0, -1, -2, -3, -4
LORA_ECUDA, LORA_ENOMEM, LORA_ESTATE, LORA_ETIMEOUT = -5, -6, -7, -8
LORA_ENOENT, LORA_ECAPACITY, LORA_EBOUNDS = -9, -10, -11

# every entry point declared in include/lora_layer.h
ABI_FUNCTIONS = ("lora_layer_create", "lora_layer_create_pooled", "lora_layer_create_fp8",
                 "lora_get_pool_usage",
                 "load_adapter_slot", "load_adapter_slot_composed",
                 "unload_adapter_slot",
                 "set_batch_segments", "lora_forward", "lora_forward_host", "lora_get_status",
                 "lora_get_segments", "lora_set_trace_events", "lora_set_gemm_plan",
                 "lora_last_error", "lora_layer_destroy", "lora_build_segments_static",
                 "lora_wait_selftest", "lora_get_launch_count")
# every entry point declared in include/lora_residency.h
CACHE_FUNCTIONS = ("lora_cache_create", "lora_cache_add", "lora_cache_add_composed",
                   "lora_cache_remove",
                   "lora_cache_map_batch", "lora_cache_prefetch", "lora_cache_slot_of",
                   "lora_cache_get_stats", "lora_cache_stream", "lora_cache_sync",
                   "lora_cache_last_error", "lora_cache_destroy")


class CacheStats(ctypes.Structure):
    """lora_cache_stats_t."""
    _fields_ = [("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("prefetches", ctypes.c_int64), ("gpu_evictions", ctypes.c_int64),
                ("host_evictions", ctypes.c_int64), ("bytes_swapped", ctypes.c_int64),
                ("resident", ctypes.c_int32), ("registered", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


class LoraError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        self.code = code
        super().__init__("%s (%d)%s" % (STATUS.get(code, "?"), code, ": " + msg if msg else ""))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is not built (run __graft_entry__.build() or python -m "
                          "segmented_rank_gemm_gb300.build [--debug]); no fallback exists"
                          % os.path.basename(LIB_PATH))
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.lora_layer_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, vp, vp]
    L.lora_layer_create_pooled.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, vp,
                                           vp, i32]
    L.lora_get_pool_usage.argtypes = [vp, vp, vp]
    L.lora_layer_create_fp8.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, vp, vp]
    L.load_adapter_slot.argtypes = [vp, i32, vp, vp, i32, f32, vp]
    L.load_adapter_slot_composed.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.unload_adapter_slot.argtypes = [vp, i32, vp]
    L.set_batch_segments.argtypes = [vp, vp, i32, vp]
    L.lora_forward.argtypes = [vp, vp, vp, i32, vp]
    L.lora_forward_host.argtypes = [vp, vp, vp, vp, i32, vp]
    L.lora_get_status.argtypes = [vp, vp]
    L.lora_get_segments.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.lora_set_trace_events.argtypes = [vp, vp]
    L.lora_set_gemm_plan.argtypes = [vp, i32, i32, i32]
    L.lora_build_segments_static.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.lora_wait_selftest.argtypes = [i32, vp]
    L.lora_get_launch_count.argtypes = [vp]
    L.lora_last_error.argtypes = [vp]
    L.lora_last_error.restype = ctypes.c_char_p
    L.lora_layer_destroy.argtypes = [vp]
    L.lora_layer_destroy.restype = None
    for name in ABI_FUNCTIONS:
        if name not in ("lora_last_error", "lora_layer_destroy"):
            getattr(L, name).restype = i32
    i64 = ctypes.c_int64
    L.lora_cache_create.argtypes = [ctypes.POINTER(vp), vp, i32, i32, i32]
    L.lora_cache_add.argtypes = [vp, i64, i32, f32, vp, vp]
    L.lora_cache_add_composed.argtypes = [vp, i64, i32, vp, vp]
    L.lora_cache_remove.argtypes = [vp, i64]
    L.lora_cache_map_batch.argtypes = [vp, vp, i32, vp, vp]
    L.lora_cache_prefetch.argtypes = [vp, vp, i32]
    L.lora_cache_slot_of.argtypes = [vp, i64]
    L.lora_cache_get_stats.argtypes = [vp, ctypes.POINTER(CacheStats)]
    L.lora_cache_stream.argtypes = [vp]
    L.lora_cache_stream.restype = vp
    L.lora_cache_sync.argtypes = [vp]
    L.lora_cache_last_error.argtypes = [vp]
    L.lora_cache_last_error.restype = ctypes.c_char_p
    L.lora_cache_destroy.argtypes = [vp]
    L.lora_cache_destroy.restype = None
    for name in ("lora_cache_create", "lora_cache_add", "lora_cache_add_composed",
                 "lora_cache_remove",
                 "lora_cache_map_batch", "lora_cache_prefetch", "lora_cache_slot_of",
                 "lora_cache_get_stats", "lora_cache_sync"):
        getattr(L, name).restype = i32
    return L


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _check(handle, rc: int) -> int:
    if rc < 0:
        msg = _lib.lora_last_error(handle).decode() if handle else ""
        raise LoraError(rc, msg)
    return rc


def dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return LORA_BF16
    if dtype == torch.float32:
        return LORA_F32
    raise ValueError("unsupported dtype %s (bf16 or fp32)" % dtype)


# ---------------------------------------------------------------------------------
# C names
# ---------------------------------------------------------------------------------

def lora_layer_create(K, N, num_slots, max_rank, max_tokens, dtype, W, stream=None) -> int:
    h = ctypes.c_void_p()
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    _check(None, _lib.lora_layer_create(ctypes.byref(h), K, N, num_slots, max_rank, max_tokens,
                                        code, _ptr(W), _stream(stream)))
    return h.value


def lora_layer_create_pooled(K, N, num_slots, max_rank, max_tokens, dtype, W, pool_rows,
                             stream=None) -> int:
    h = ctypes.c_void_p()
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    _check(None, _lib.lora_layer_create_pooled(ctypes.byref(h), K, N, num_slots, max_rank,
                                               max_tokens, code, _ptr(W), _stream(stream),
                                               int(pool_rows)))
    return h.value


def lora_layer_create_fp8(K, N, num_slots, max_rank, max_tokens, W, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(None, _lib.lora_layer_create_fp8(ctypes.byref(h), K, N, num_slots, max_rank,
                                            max_tokens, _ptr(W), _stream(stream)))
    return h.value


def lora_get_pool_usage(layer):
    """(rows in use, rows in the pool)."""
    used, total = ctypes.c_int(), ctypes.c_int()
    _check(layer, _lib.lora_get_pool_usage(layer, ctypes.byref(used), ctypes.byref(total)))
    return used.value, total.value


def load_adapter_slot(layer, slot, A, B, r, alpha, side_stream=None) -> None:
    _check(layer, _lib.load_adapter_slot(layer, slot, _ptr(A), _ptr(B), r, float(alpha),
                                         _stream(side_stream)))


def load_adapter_slot_composed(layer, slot, members, side_stream=None) -> None:
    """``members``: list of (A [K, r], B [r, N], alpha, weight) tensors/values."""
    n = len(members)
    A = (ctypes.c_void_p * n)(*[_ptr(m[0]) for m in members])
    B = (ctypes.c_void_p * n)(*[_ptr(m[1]) for m in members])
    r = (ctypes.c_int * n)(*[int(m[0].shape[1]) for m in members])
    al = (ctypes.c_float * n)(*[float(m[2]) for m in members])
    w = (ctypes.c_float * n)(*[float(m[3]) for m in members])
    _check(layer, _lib.load_adapter_slot_composed(
        layer, slot, n, ctypes.cast(A, ctypes.c_void_p), ctypes.cast(B, ctypes.c_void_p),
        ctypes.cast(r, ctypes.c_void_p), ctypes.cast(al, ctypes.c_void_p),
        ctypes.cast(w, ctypes.c_void_p), _stream(side_stream)))


def unload_adapter_slot(layer, slot, side_stream=None) -> None:
    _check(layer, _lib.unload_adapter_slot(layer, slot, _stream(side_stream)))


def set_batch_segments(layer, token_slot, T, stream=None) -> None:
    _check(layer, _lib.set_batch_segments(layer, _ptr(token_slot), T, _stream(stream)))


def lora_forward(layer, x, y, T, stream=None) -> None:
    _check(layer, _lib.lora_forward(layer, _ptr(x), _ptr(y), T, _stream(stream)))


def lora_forward_host(layer, x_host, token_slot_host, y_host, T, stream=None) -> None:
    _check(layer, _lib.lora_forward_host(layer, _ptr(x_host), _ptr(token_slot_host),
                                         _ptr(y_host), T, _stream(stream)))


def lora_get_status(layer, stream=None) -> int:
    """Returns the status code (LORA_OK, LORA_EID, LORA_ETIMEOUT) without raising."""
    return _lib.lora_get_status(layer, _stream(stream))


def lora_get_segments(layer, max_tokens, num_slots, stream=None):
    import numpy as np
    perm = np.zeros(max(max_tokens, 1), np.int32)
    offs = np.zeros(num_slots + 1, np.int32)
    sslot = np.zeros(num_slots, np.int32)
    n_seg, n_ad = ctypes.c_int32(), ctypes.c_int32()
    _check(layer, _lib.lora_get_segments(layer, perm.ctypes.data, offs.ctypes.data,
                                         sslot.ctypes.data, ctypes.addressof(n_seg),
                                         ctypes.addressof(n_ad), _stream(stream)))
    g, t_a = n_seg.value, n_ad.value
    return perm[:t_a].copy(), offs[:g + 1].copy(), sslot[:g].copy()


def lora_set_trace_events(layer, events) -> None:
    """``events``: None, or 6 ``torch.cuda.Event(enable_timing=True)`` objects."""
    if events is None:
        _check(layer, _lib.lora_set_trace_events(layer, None))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * 6)(*[e.cuda_event for e in events])
    _check(layer, _lib.lora_set_trace_events(layer, ctypes.cast(arr, ctypes.c_void_p)))


def lora_set_gemm_plan(layer, block_n: int, k_split: int = 1, cta_pair: int = 0) -> None:
    """Fix the base GEMM's N tile, K split and CTA pairing; ``block_n=0`` restores the
    automatic plan."""
    _check(layer, _lib.lora_set_gemm_plan(layer, int(block_n), int(k_split), int(cta_pair)))


def lora_build_segments_static(token_slot, T, num_slots, slot_loaded, perm, seg_offsets,
                               seg_slot, counts, stream=None) -> None:
    """Segment builder without any device allocation (scratch in a static device array);
    all tensors are caller-owned CUDA int32 tensors, ``slot_loaded`` may be None.

    The C entry point cannot see buffer sizes, so an undersized tensor here would become
    an out-of-bounds device write: each tensor is checked first (int32, on a CUDA device,
    contiguous, at least perm >= T, seg_offsets >= num_slots + 1, seg_slot >= num_slots,
    counts >= 3, token_slot >= T, slot_loaded >= num_slots) and LORA_EINVAL is raised
    otherwise."""
    T, num_slots = int(T), int(num_slots)
    need = {"token_slot": (token_slot, T), "perm": (perm, T),
            "seg_offsets": (seg_offsets, num_slots + 1), "seg_slot": (seg_slot, num_slots),
            "counts": (counts, 3)}
    if slot_loaded is not None:
        need["slot_loaded"] = (slot_loaded, num_slots)
    for name, (t, n) in need.items():
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda
                or not t.is_contiguous() or t.numel() < max(n, 0)):
            raise LoraError(LORA_EINVAL, "lora_build_segments_static: %s must be a contiguous "
                            "CUDA int32 tensor of at least %d elements" % (name, n))
    rc = _lib.lora_build_segments_static(_ptr(token_slot), T, num_slots, _ptr(slot_loaded),
                                         _ptr(perm), _ptr(seg_offsets), _ptr(seg_slot),
                                         _ptr(counts), _stream(stream))
    if rc < 0:
        raise LoraError(rc, "lora_build_segments_static")


def lora_wait_selftest(which: int, stream=None) -> int:
    """Run one bounded wait that nothing completes; returns the status (LORA_ETIMEOUT is
    the expected result) without raising."""
    return _lib.lora_wait_selftest(int(which), _stream(stream))


def lora_get_launch_count(layer) -> int:
    """Kernels the layer launched since its last set_batch_segments."""
    return int(_lib.lora_get_launch_count(layer))


def lora_last_error(layer) -> str:
    return _lib.lora_last_error(layer).decode()


def lora_layer_destroy(layer) -> None:
    _lib.lora_layer_destroy(layer)


# ---------------------------------------------------------------------------------
# owner object
# ---------------------------------------------------------------------------------

class LoraLayer:
    """Owns one C layer.  ``W`` [K, N] is a CUDA tensor (bf16 or fp32)."""

    def __init__(self, W: torch.Tensor, num_slots: int, max_rank: int, max_tokens: int,
                 stream=None, pool_rows: int = 0, fp8_base: bool = False):
        """``pool_rows`` > 0: adapters stored at their true rank in a row pool of that many
        rank rows (lora_layer_create_pooled); ``fp8_base``: the base product in e4m3
        (lora_layer_create_fp8; W bf16)."""
        if not W.is_cuda:
            raise ValueError("W must be a CUDA tensor")
        self.K, self.N = int(W.shape[0]), int(W.shape[1])
        self.num_slots, self.max_rank, self.max_tokens = num_slots, max_rank, max_tokens
        self.dtype = W.dtype
        if fp8_base:
            if pool_rows or W.dtype != torch.bfloat16:
                raise ValueError("an e4m3 base layer takes a bf16 W and no row pool")
            self.handle = lora_layer_create_fp8(self.K, self.N, num_slots, max_rank, max_tokens,
                                                W.contiguous(), stream)
        elif pool_rows:
            self.handle = lora_layer_create_pooled(self.K, self.N, num_slots, max_rank,
                                                   max_tokens, W.dtype, W.contiguous(),
                                                   pool_rows, stream)
        else:
            self.handle = lora_layer_create(self.K, self.N, num_slots, max_rank, max_tokens,
                                            W.dtype, W.contiguous(), stream)
        self._keep = {}

    def load(self, slot: int, A: torch.Tensor, B: torch.Tensor, alpha: float, side_stream=None):
        A, B = A.contiguous(), B.contiguous()
        if A.dtype != self.dtype or B.dtype != self.dtype:
            raise ValueError("adapter dtype must match the layer dtype")
        r = int(A.shape[1])
        if tuple(A.shape) != (self.K, r) or tuple(B.shape) != (r, self.N):
            raise ValueError("A must be [K, r] and B [r, N]")
        load_adapter_slot(self.handle, slot, A, B, r, alpha, side_stream)
        self._keep[slot] = (A, B)  # keep sources alive until the copy has run

    def load_composed(self, slot: int, members, side_stream=None):
        """``members``: list of (A [K, r_i], B [r_i, N], alpha_i, weight_i)."""
        members = [(A.contiguous(), B.contiguous(), alpha, w) for A, B, alpha, w in members]
        for A, B, _, _ in members:
            if A.dtype != self.dtype or B.dtype != self.dtype:
                raise ValueError("adapter dtype must match the layer dtype")
            r = int(A.shape[1])
            if tuple(A.shape) != (self.K, r) or tuple(B.shape) != (r, self.N):
                raise ValueError("A must be [K, r] and B [r, N]")
        load_adapter_slot_composed(self.handle, slot, members, side_stream)
        self._keep[slot] = members  # keep sources alive until the copies have run

    def unload(self, slot: int, side_stream=None):
        unload_adapter_slot(self.handle, slot, side_stream)

    def set_batch(self, token_slot: torch.Tensor, stream=None):
        if token_slot.dtype != torch.int32 or not token_slot.is_cuda:
            raise ValueError("token_slot must be a CUDA int32 tensor")
        self._ids = token_slot
        set_batch_segments(self.handle, token_slot, int(token_slot.shape[0]), stream)

    def forward(self, x: torch.Tensor, y: torch.Tensor = None, stream=None) -> torch.Tensor:
        if x.dtype != self.dtype or not x.is_cuda:
            raise ValueError("x must be a CUDA tensor of the layer dtype")
        T = int(x.shape[0])
        if y is None:
            y = torch.empty(T, self.N, dtype=self.dtype, device=x.device)
        lora_forward(self.handle, x, y, T, stream)
        return y

    def __call__(self, x, token_slot, y=None, stream=None):
        self.set_batch(token_slot, stream)
        return self.forward(x, y, stream)

    def forward_host(self, x_host, ids_host, y_host, stream=None):
        lora_forward_host(self.handle, x_host, ids_host, y_host, int(x_host.shape[0]), stream)
        return y_host

    def launch_count(self) -> int:
        return lora_get_launch_count(self.handle)

    def status(self, stream=None) -> int:
        return lora_get_status(self.handle, stream)

    def segments(self, stream=None):
        return lora_get_segments(self.handle, self.max_tokens, self.num_slots, stream)

    def pool_usage(self):
        """(rank rows in use, rank rows in the pool)."""
        return lora_get_pool_usage(self.handle)

    def set_gemm_plan(self, block_n: int, k_split: int = 1, cta_pair: int = 0):
        lora_set_gemm_plan(self.handle, block_n, k_split, cta_pair)

    def close(self):
        if getattr(self, "handle", None):
            lora_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------------------------
# adapter cache (include/lora_residency.h)
# ---------------------------------------------------------------------------------

def _check_cache(cache, rc: int) -> int:
    if rc < 0:
        msg = _lib.lora_cache_last_error(cache).decode() if cache else ""
        raise LoraError(rc, msg)
    return rc


def lora_cache_create(layers, num_slots: int, host_capacity: int) -> int:
    """``layers``: layer handles (ints) or ``LoraLayer`` objects; [] keeps only the books."""
    hs = [l.handle if isinstance(l, LoraLayer) else l for l in layers]
    arr = (ctypes.c_void_p * max(len(hs), 1))(*hs)
    h = ctypes.c_void_p()
    _check_cache(None, _lib.lora_cache_create(ctypes.byref(h), ctypes.cast(arr, ctypes.c_void_p)
                                              if hs else None, len(hs), num_slots,
                                              host_capacity))
    return h.value


def lora_cache_add(cache, adapter_id: int, r: int, alpha: float, A_host=(), B_host=()) -> None:
    """``A_host`` / ``B_host``: per layer, contiguous CPU tensors [K, r] / [r, N]."""
    n = len(A_host)
    A = (ctypes.c_void_p * max(n, 1))(*[_ptr(a) for a in A_host])
    B = (ctypes.c_void_p * max(n, 1))(*[_ptr(b) for b in B_host])
    _check_cache(cache, _lib.lora_cache_add(cache, int(adapter_id), int(r), float(alpha),
                                            ctypes.cast(A, ctypes.c_void_p) if n else None,
                                            ctypes.cast(B, ctypes.c_void_p) if n else None))


def lora_cache_add_composed(cache, adapter_id: int, member_ids, weights) -> None:
    import numpy as np
    m = np.ascontiguousarray(member_ids, dtype=np.int64)
    w = np.ascontiguousarray(weights, dtype=np.float32)
    if m.shape != w.shape:
        raise ValueError("one weight per member")
    _check_cache(cache, _lib.lora_cache_add_composed(cache, int(adapter_id), len(m),
                                                     m.ctypes.data if len(m) else None,
                                                     w.ctypes.data if len(w) else None))


def lora_cache_remove(cache, adapter_id: int) -> None:
    _check_cache(cache, _lib.lora_cache_remove(cache, int(adapter_id)))


def lora_cache_map_batch(cache, token_adapter, stream=0):
    """``token_adapter``: int64 numpy array (host); returns the int32 numpy slot ids.
    ``stream``: the batches' stream (a torch stream, a handle, or None for torch's current
    stream; the default 0 is the legacy default stream, as a cache without layers needs)."""
    import numpy as np
    ta = np.ascontiguousarray(token_adapter, dtype=np.int64)
    out = np.empty(max(len(ta), 1), np.int32)
    _check_cache(cache, _lib.lora_cache_map_batch(cache, ta.ctypes.data, len(ta),
                                                  out.ctypes.data, _stream(stream)))
    return out[:len(ta)]


def lora_cache_prefetch(cache, ids) -> None:
    import numpy as np
    a = np.ascontiguousarray(ids, dtype=np.int64)
    _check_cache(cache, _lib.lora_cache_prefetch(cache, a.ctypes.data if len(a) else None,
                                                 len(a)))


def lora_cache_slot_of(cache, adapter_id: int) -> int:
    return _lib.lora_cache_slot_of(cache, int(adapter_id))


def lora_cache_get_stats(cache) -> dict:
    st = CacheStats()
    _check_cache(cache, _lib.lora_cache_get_stats(cache, ctypes.byref(st)))
    return st.as_dict()


def lora_cache_stream(cache) -> int:
    return _lib.lora_cache_stream(cache) or 0


def lora_cache_sync(cache) -> None:
    _check_cache(cache, _lib.lora_cache_sync(cache))


def lora_cache_last_error(cache) -> str:
    return _lib.lora_cache_last_error(cache).decode()


def lora_cache_destroy(cache) -> None:
    _lib.lora_cache_destroy(cache)


class AdapterCache:
    """Owns one adapter cache over ``layers`` (``LoraLayer`` objects, kept alive here)."""

    def __init__(self, layers, num_slots: int, host_capacity: int):
        self.layers = list(layers)
        self.num_slots, self.host_capacity = num_slots, host_capacity
        self.handle = lora_cache_create(self.layers, num_slots, host_capacity)

    def add(self, adapter_id: int, A_list, B_list, alpha: float, r: int = None) -> None:
        """Per layer: A [K, r] and B [r, N] in the layer dtype (moved to host memory)."""
        A_list = [a.detach().to("cpu").contiguous() for a in A_list]
        B_list = [b.detach().to("cpu").contiguous() for b in B_list]
        for L, A, B in zip(self.layers, A_list, B_list):
            if A.dtype != L.dtype or B.dtype != L.dtype:
                raise ValueError("adapter dtype must match the layer dtype")
            if A.shape[0] != L.K or B.shape[1] != L.N or A.shape[1] != B.shape[0]:
                raise ValueError("A must be [K, r] and B [r, N]")
        if r is None:
            r = int(A_list[0].shape[1])
        lora_cache_add(self.handle, adapter_id, r, alpha, A_list, B_list)

    def add_composed(self, adapter_id: int, member_ids, weights) -> None:
        lora_cache_add_composed(self.handle, adapter_id, member_ids, weights)

    def remove(self, adapter_id: int) -> None:
        lora_cache_remove(self.handle, adapter_id)

    def map_batch(self, token_adapter, stream=None):
        return lora_cache_map_batch(self.handle, token_adapter, stream)

    def prefetch(self, ids) -> None:
        lora_cache_prefetch(self.handle, ids)

    def slot_of(self, adapter_id: int) -> int:
        return lora_cache_slot_of(self.handle, adapter_id)

    def stats(self) -> dict:
        return lora_cache_get_stats(self.handle)

    @property
    def stream(self) -> int:
        return lora_cache_stream(self.handle)

    def sync(self) -> None:
        lora_cache_sync(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            lora_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
