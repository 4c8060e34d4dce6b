"""CPU fp64 oracle for the mixed-adapter LoRA linear layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA path and never imports it.

The arithmetic lives in ``lora_oracle.c`` (plain C loops in double precision, OpenMP
over rows); this module only compiles it with gcc and marshals numpy arrays.

Definition (the pages' statement of the layer, see the C file's header for the
sections it follows)::

    y[i] = x[i] W + [slot_i != -1] * (alpha_s / r_s) * (x[i] A_s) B_s,   s = slot_i

Adapters are given as a slot table: per slot an ``A`` of shape ``[K, r]``, a ``B`` of
shape ``[r, N]`` and ``alpha``; empty slots are ``None``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .sizes import adapter_params, adapter_bytes, lora_flop_share  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_lora_oracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile ``lora_oracle.c`` into ``_lora_oracle.so`` (plain gcc, no CUDA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.run(["gcc", *GCC_FLAGS, _SRC, "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_variant(src_text: str, out_path: str) -> ctypes.CDLL:
    """Compile a modified copy of the oracle source (used by the tests that plant a
    mistake in the oracle to show that its pins catch it)."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *GCC_FLAGS, src_path, "-o", out_path], check=True)
    return _bind(ctypes.CDLL(out_path))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64, dp, ip = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_num_threads.argtypes = [i32]
    lib.oracle_segments.restype = i32
    lib.oracle_segments.argtypes = [i32, ip, i32, ip, ip, ip, ip]
    lib.oracle_forward_rows.restype = None
    lib.oracle_forward_rows.argtypes = [i32, i32, i32, i32, i32, dp, dp, dp, dp, ip, dp, ip,
                                        i32, ip, dp]
    lib.oracle_forward_grouped.restype = i32
    lib.oracle_forward_grouped.argtypes = [i32, i32, i32, i32, i32, dp, dp, dp, dp, ip, dp, ip, dp]
    lib.oracle_forward_merged.restype = None
    lib.oracle_forward_merged.argtypes = [i32, i32, i32, i32, i32, dp, dp, dp, dp, ip, dp, ip, dp]
    del i64
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: exact widening of bf16 / fp32 values
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class SlotTable:
    """Adapters packed as dense fp64 arrays for the C oracle.

    ``adapters`` is a list of length S whose entries are ``None`` (empty slot) or a
    tuple ``(A [K, r], B [r, N], alpha)``.  Padding columns/rows beyond each true rank
    are zero and never read by the oracle.
    """

    def __init__(self, adapters, K: int, N: int):
        self.S = len(adapters)
        ranks = [a[0].shape[1] for a in adapters if a is not None]
        self.R = max(ranks) if ranks else 1
        self.K, self.N = K, N
        self.A = np.zeros((self.S, K, self.R), dtype=np.float64)
        self.B = np.zeros((self.S, self.R, N), dtype=np.float64)
        self.rank = np.ones(self.S, dtype=np.int32)
        self.alpha = np.zeros(self.S, dtype=np.float64)
        self.present = np.zeros(self.S, dtype=bool)
        for s, ad in enumerate(adapters):
            if ad is None:
                continue
            A, B, alpha = ad
            A, B = _f64(A), _f64(B)
            r = A.shape[1]
            assert A.shape == (K, r) and B.shape == (r, N), (A.shape, B.shape)
            self.A[s, :, :r] = A
            self.B[s, :r, :] = B
            self.rank[s] = r
            self.alpha[s] = float(alpha)
            self.present[s] = True


def segments(slot, S: int, _lib=None):
    """Reference segment builder: returns (perm, seg_offsets, seg_slot, n_bad)."""
    L = _lib or lib()
    slot = _i32(slot)
    T = slot.shape[0]
    perm = np.zeros(max(T, 1), dtype=np.int32)
    offs = np.zeros(S + 1, dtype=np.int32)
    sslot = np.zeros(max(S, 1), dtype=np.int32)
    n_seg = np.zeros(1, dtype=np.int32)
    bad = L.oracle_segments(T, _ptr(slot), S, _ptr(perm), _ptr(offs), _ptr(sslot), _ptr(n_seg))
    g = int(n_seg[0])
    t_a = int(offs[g]) if g > 0 else 0
    return perm[:t_a].copy(), offs[:g + 1].copy(), sslot[:g].copy(), int(bad)


def _common(x, W, table: SlotTable, slot):
    x, W, slot = _f64(x), _f64(W), _i32(slot)
    T, K = x.shape
    K2, N = W.shape
    assert K == K2 == table.K and N == table.N and slot.shape == (T,)
    return x, W, slot, T, K, N


def forward_rows(x, W, table: SlotTable, slot, rows=None, _lib=None) -> np.ndarray:
    """Evaluator 1 (row by row).  ``rows`` selects a subset; returns [len(rows), N]."""
    L = _lib or lib()
    x, W, slot, T, K, N = _common(x, W, table, slot)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64))
    y = np.zeros((rows.shape[0], N), dtype=np.float64)
    L.oracle_forward_rows(T, K, N, table.S, table.R, _ptr(x), _ptr(W), _ptr(table.A),
                          _ptr(table.B), _ptr(table.rank), _ptr(table.alpha), _ptr(slot),
                          rows.shape[0], _ptr(rows), _ptr(y))
    return y


def forward_grouped(x, W, table: SlotTable, slot, _lib=None) -> np.ndarray:
    """Evaluator 2 (shared base product + one small product per segment)."""
    L = _lib or lib()
    x, W, slot, T, K, N = _common(x, W, table, slot)
    y = np.zeros((T, N), dtype=np.float64)
    L.oracle_forward_grouped(T, K, N, table.S, table.R, _ptr(x), _ptr(W), _ptr(table.A),
                             _ptr(table.B), _ptr(table.rank), _ptr(table.alpha), _ptr(slot),
                             _ptr(y))
    return y


def forward_merged(x, W, table: SlotTable, slot, _lib=None) -> np.ndarray:
    """Evaluator 3 (x times the merged weight W + (alpha/r) A B of each row's adapter)."""
    L = _lib or lib()
    x, W, slot, T, K, N = _common(x, W, table, slot)
    y = np.zeros((T, N), dtype=np.float64)
    L.oracle_forward_merged(T, K, N, table.S, table.R, _ptr(x), _ptr(W), _ptr(table.A),
                            _ptr(table.B), _ptr(table.rank), _ptr(table.alpha), _ptr(slot),
                            _ptr(y))
    return y


def forward_composed(x, W, compositions, slot) -> np.ndarray:
    """Rows whose slot holds a composition of adapters ("Multi-LoRA Serving 与 Adapter
    隔离", adapter ownership in a continuous batch: a request may compose several LoRAs,
    which are added, identified by the ordered members and their weights):

        y[i] = x[i] W + sum_m weight_m * (alpha_m / r_m) * (x[i] A_m) B_m,   m in slot_i

    ``compositions``: per slot ``None`` (empty) or a list of members
    ``(A [K, r_m], B [r_m, N], alpha_m, weight_m)``.  Rows with slot -1, outside the list or
    naming an empty slot are base only.  fp64 from the exact input values; numpy's matmul
    serves as the dense product, nothing else is fused or reordered.
    """
    x, W, slot = _f64(x), _f64(W), _i32(slot)
    y = x @ W
    for s, comp in enumerate(compositions):
        if not comp:
            continue
        rows = np.nonzero(slot == s)[0]
        if rows.size == 0:
            continue
        xs = x[rows]
        for A, B, alpha, weight in comp:
            A, B = _f64(A), _f64(B)
            r = A.shape[1]
            y[rows] += float(weight) * (float(alpha) / r) * ((xs @ A) @ B)
    return y
