"""Mixed-adapter LoRA linear layer (SGMV / BGMV) for GB300 (sm_103a).

y = x W + (alpha_s / r_s) * (x A_s) B_s per token row, s = the row's adapter slot
(-1 = base only).  The compute runs in the CUDA library ``liblora_layer.so`` behind the
C ABI declared in ``include/lora_layer.h``; ``segmented_rank_gemm_gb300.lora`` is the
thin ctypes binding with the same names.  Importing the binding raises if the library
has not been built: there is no CPU fallback.

``segmented_rank_gemm_gb300.workloads`` (seeded synthetic inputs) imports without the
library.
"""
import importlib

__all__ = ["lora", "workloads", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
