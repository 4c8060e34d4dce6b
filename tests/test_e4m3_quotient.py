"""The e4m3 row quantiser's fast quotient takes the same e4m3 decision as the correctly
rounded division on every input it can meet (exhaustive, on the host).

The kernel divides each element of a row by the row's scale with a reciprocal and one FMA
correction instead of a full division; the decision that matters is the e4m3 value of the
quotient (the oracle rounds RN(x / s) to e4m3).  tests/e4m3_quotient_check.c enumerates
every bf16 row maximum whose scale is in the fast range and every bf16 element up to it
(about 4.9e8 pairs, ~30 s) and counts the pairs whose e4m3 values differ.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_fast_quotient_takes_the_division_s_e4m3_decisions(tmp_path):
    exe = str(tmp_path / "e4m3_quotient_check")
    # strict IEEE single precision: no contraction of the product into the FMA
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "e4m3_quotient_check.c"), "-lm"], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
    m = re.search(r"pairs (\d+) quotient_mismatches (\d+) e4m3_mismatches (\d+)", out)
    assert m, out
    pairs, _, e4m3_bad = (int(g) for g in m.groups())
    assert pairs > 4 * 10**8, out
    assert e4m3_bad == 0, out
