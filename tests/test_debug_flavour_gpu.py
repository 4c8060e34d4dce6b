"""The debug flavour of the library (``liblora_layer_debug.so``, built with -DLORA_DEBUG).

Its kernels check every index they take from data -- the slot rows of the adapter pools,
the rows of the fp32 delta and v buffers, the K-split planes of v -- and, instead of
accessing memory outside a buffer, skip the access and raise a device flag that
``lora_get_status`` reports as LORA_EBOUNDS.  Nothing traps.

The test builds that flavour, then runs the edge-case GPU suites (ragged shapes, empty and
single-row batches, every GEMM tiling, pooled and composed slots, e4m3 base, the builder,
the adapter cache) in a child process that loads it (LORA_LAYER_LIBRARY=debug).  Those
suites check ``status() == LORA_OK`` (or the id error they plant) after their forwards, so
any bounds flag fails them; the child also reports which library it loaded.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EDGE_SUITES = ["tests/test_forward_gpu.py", "tests/test_gemm_plans_gpu.py",
               "tests/test_pooled_gpu.py", "tests/test_composition_gpu.py",
               "tests/test_builder_gpu.py", "tests/test_fp8_gpu.py",
               "tests/test_residency_gpu.py", "tests/test_vmode_gpu.py"]


def test_debug_flavour_flags_stay_clean_on_the_edge_case_suites():
    from segmented_rank_gemm_gb300 import build as b
    path = b.build(debug=True)
    assert os.path.basename(path) == "liblora_layer_debug.so"
    env = dict(os.environ, LORA_LAYER_LIBRARY="debug")
    which = subprocess.run(
        [sys.executable, "-c", "from segmented_rank_gemm_gb300 import lora; print(lora.LIB_PATH)"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert which.returncode == 0, which.stderr[-2000:]
    assert which.stdout.strip().endswith("liblora_layer_debug.so"), which.stdout
    run = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
         *EDGE_SUITES], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert run.returncode == 0, run.stdout[-4000:] + run.stderr[-2000:]
    assert " passed" in run.stdout
