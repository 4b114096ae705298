"""Plant known mistakes in the oracle (on the CPU) and check that its pins
catch every one: each mutant is the oracle compiled with ORACLE_MUTANT=k,
and the pin suite tests/test_oracle.py must fail against it."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    1: "sm_scale dropped from the scores",
    2: "P.V multiplies K instead of V",
    3: "output not divided by the weight sum",
    4: "lse in log2 instead of ln",
    5: "q head h reads kv head h % Hk instead of h / group",
    6: "last_page_len ignored (last page taken as full)",
    7: "rows of a page read in reverse",
    8: "append writes slot last_page_len instead of last_page_len - 1",
    9: "merge weights exp(L - lse_c) instead of exp(lse_c - L)",
    10: "contiguous append one row early",
    11: "NHD cache addressed as HND",
    12: "E4M3 exponent bias 8 instead of 7",
    13: "FP8 V scaled by the K scale",
    14: "E4M3 exponent field 0 decoded as a normal number",
    15: "E4M3 rounding ties away from zero instead of to the even code",
    16: "E4M3 rounding overflows to NaN instead of saturating at 448",
    17: "FP8 append multiplies by the K scale instead of dividing",
    18: "empty request gives lse 0 instead of -inf",
    19: "contiguous decode reads max_kv_len rows instead of valid_kv_len",
    20: "merge normalises by the largest lse instead of the log-sum-exp",
}


@pytest.mark.parametrize("k", sorted(MUTANTS))
def test_pins_catch_mutant(k, tmp_path):
    so = tmp_path / f"liboracle_mutant{k}.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                           f"-DORACLE_MUTANT={k}", SRC, "-o", str(so)])
    env = dict(os.environ, PD_ORACLE_LIBRARY=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught mutant {k} ({MUTANTS[k]}):\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:]
