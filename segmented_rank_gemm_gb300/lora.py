"""ctypes binding of the layer's C ABI (``include/lora_layer.h``).

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

from .build import LIB_PATH

LORA_F32, LORA_BF16 = 0, 1
STATUS = {0: "LORA_OK", -1: "LORA_EINVAL", -2: "LORA_ESLOT", -3: "LORA_ERANK", -4: "LORA_EID",
          -5: "LORA_ECUDA", -6: "LORA_ENOMEM", -7: "LORA_ESTATE", -8: "LORA_ETIMEOUT"}
LORA_OK, LORA_EINVAL, LORA_ESLOT, LORA_ERANK, LORA_EID = 0, -1, -2, -3, -4
LORA_ECUDA, LORA_ENOMEM, LORA_ESTATE, LORA_ETIMEOUT = -5, -6, -7, -8

# every entry point declared in include/lora_layer.h
ABI_FUNCTIONS = ("lora_layer_create", "load_adapter_slot", "unload_adapter_slot",
                 "set_batch_segments", "lora_forward", "lora_forward_host", "lora_get_status",
                 "lora_get_segments", "lora_set_trace_events", "lora_set_gemm_plan",
                 "lora_last_error", "lora_layer_destroy", "lora_build_segments_static")


class LoraError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        self.code = code
        super().__init__("%s (%d)%s" % (STATUS.get(code, "?"), code, ": " + msg if msg else ""))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("liblora_layer.so is not built (run __graft_entry__.build() or "
                          "python -m segmented_rank_gemm_gb300.build); no fallback exists")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.lora_layer_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, vp, vp]
    L.load_adapter_slot.argtypes = [vp, i32, vp, vp, i32, f32, vp]
    L.unload_adapter_slot.argtypes = [vp, i32, vp]
    L.set_batch_segments.argtypes = [vp, vp, i32, vp]
    L.lora_forward.argtypes = [vp, vp, vp, i32, vp]
    L.lora_forward_host.argtypes = [vp, vp, vp, vp, i32, vp]
    L.lora_get_status.argtypes = [vp, vp]
    L.lora_get_segments.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.lora_set_trace_events.argtypes = [vp, vp]
    L.lora_set_gemm_plan.argtypes = [vp, i32, i32, i32]
    L.lora_build_segments_static.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.lora_last_error.argtypes = [vp]
    L.lora_last_error.restype = ctypes.c_char_p
    L.lora_layer_destroy.argtypes = [vp]
    L.lora_layer_destroy.restype = None
    for name in ABI_FUNCTIONS:
        if name not in ("lora_last_error", "lora_layer_destroy"):
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


def load_adapter_slot(layer, slot, A, B, r, alpha, side_stream=None) -> None:
    _check(layer, _lib.load_adapter_slot(layer, slot, _ptr(A), _ptr(B), r, float(alpha),
                                         _stream(side_stream)))


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
    all tensors are caller-owned CUDA int32 tensors, ``slot_loaded`` may be None."""
    rc = _lib.lora_build_segments_static(_ptr(token_slot), T, num_slots, _ptr(slot_loaded),
                                         _ptr(perm), _ptr(seg_offsets), _ptr(seg_slot),
                                         _ptr(counts), _stream(stream))
    if rc < 0:
        raise LoraError(rc, "lora_build_segments_static")


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
                 stream=None):
        if not W.is_cuda:
            raise ValueError("W must be a CUDA tensor")
        self.K, self.N = int(W.shape[0]), int(W.shape[1])
        self.num_slots, self.max_rank, self.max_tokens = num_slots, max_rank, max_tokens
        self.dtype = W.dtype
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

    def status(self, stream=None) -> int:
        return lora_get_status(self.handle, stream)

    def segments(self, stream=None):
        return lora_get_segments(self.handle, self.max_tokens, self.num_slots, stream)

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
