"""The C-ABI library without a GPU: it builds, loads, exports every entry point the
header declares, and rejects bad host-side arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        names += re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from segmented_rank_gemm_gb300 import build
    build.build()
    from segmented_rank_gemm_gb300 import lora
    return lora


def test_header_declares_the_abi():
    names = header_functions()
    for n in ("lora_layer_create", "load_adapter_slot", "set_batch_segments", "lora_forward",
              "lora_layer_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in header_functions():
        assert hasattr(so, name), name
    assert set(lib.ABI_FUNCTIONS) | set(lib.CACHE_FUNCTIONS) == set(header_functions())


def test_create_rejects_bad_arguments(lib):
    L = lib.library()
    h = ctypes.c_void_p()
    dummy = 16  # never dereferenced: validation fails first
    bad = [
        (0, 8, 4, 16, 8, lib.LORA_BF16),       # K < 1
        (8, 0, 4, 16, 8, lib.LORA_BF16),       # N < 1
        (8, 8, 0, 16, 8, lib.LORA_BF16),       # no slots
        (8, 8, 5000, 16, 8, lib.LORA_BF16),    # too many slots
        (8, 8, 4, 0, 8, lib.LORA_BF16),        # rank 0
        (8, 8, 4, 129, 8, lib.LORA_BF16),      # rank above 128
        (8, 8, 4, 16, 0, lib.LORA_BF16),       # no tokens
        (12, 8, 4, 16, 8, lib.LORA_BF16),      # bf16 K not a multiple of 8
        (8, 12, 4, 16, 8, lib.LORA_BF16),      # bf16 N not a multiple of 8
        (8, 8, 4, 16, 8, 7),                   # unknown dtype
    ]
    for K, N, S, R, T, dt in bad:
        assert L.lora_layer_create(ctypes.byref(h), K, N, S, R, T, dt, dummy, None) == lib.LORA_EINVAL
        assert not h.value
    assert L.lora_layer_create(ctypes.byref(h), 8, 8, 4, 16, 8, lib.LORA_BF16, None, None) == lib.LORA_EINVAL
    assert L.lora_layer_create(None, 8, 8, 4, 16, 8, lib.LORA_BF16, dummy, None) == lib.LORA_EINVAL
    # a row pool below one slot of max_rank rows (16) or above num_slots of them (64)
    for rows in (0, 8, 65):
        assert L.lora_layer_create_pooled(ctypes.byref(h), 8, 8, 4, 16, 8, lib.LORA_BF16, dummy,
                                          None, rows) == lib.LORA_EINVAL
        assert not h.value


def test_null_layer_calls_are_rejected(lib):
    L = lib.library()
    assert L.load_adapter_slot(None, 0, 16, 16, 1, 1.0, None) == lib.LORA_EINVAL
    assert L.unload_adapter_slot(None, 0, None) == lib.LORA_EINVAL
    assert L.set_batch_segments(None, 16, 4, None) == lib.LORA_EINVAL
    assert L.lora_forward(None, 16, 32, 4, None) == lib.LORA_EINVAL
    assert L.lora_forward_host(None, 16, 16, 32, 4, None) == lib.LORA_EINVAL
    assert L.lora_get_status(None, None) == lib.LORA_EINVAL
    assert L.lora_last_error(None) == b"null layer"
    L.lora_layer_destroy(None)  # no-op


def test_no_device_is_a_cuda_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = lib.library()
    h = ctypes.c_void_p()
    rc = L.lora_layer_create(ctypes.byref(h), 64, 64, 4, 16, 8, lib.LORA_BF16, 16, None)
    assert rc in (lib.LORA_ECUDA, lib.LORA_ENOMEM) and not h.value
