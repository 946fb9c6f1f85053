"""The oracle's pins reject planted mistakes.

Each mutant is the oracle compiled with one deliberate, plausible mistake
(ORC_MUTANT in oracle/moe_oracle.c).  The pin suite is run against it in a
child process and must fail: a pin set that a dropped term, a wrong index or
a reversed tie rule passes would not pin the oracle to the pages.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    1: "bf16 rounding truncates instead of rounding to nearest even",
    2: "top-k resolves equal logits to the higher expert id",
    3: "the softmax runs over every logit instead of the k chosen",
    4: "experts are dealt to partitions round robin (e % P) instead of in blocks",
    5: "every partition slot is one too high",
    6: "the expected-copies closed form uses E - G instead of E - E/G",
    7: "the combine drops each token's last choice",
    8: "the combine ignores the router weights",
    9: "the MXFP8 block scale is one binade too high",
    10: "E2M1 rounding sends ties to the odd code",
    11: "the planner keeps a copy that ties the busiest partition",
    12: "the replica map picks the copy from the token index, not the pair's rank",
    13: "the stage-1 pre-add also takes experts of other partitions",
    14: "the NVFP4 block scale ignores the tensor scale",
}


@pytest.mark.parametrize("n", sorted(MUTANTS))
def test_pins_reject_mutant(n, tmp_path):
    lib = oracle.build_mutant(n, str(tmp_path / f"liboracle_mutant{n}.so"))
    env = dict(os.environ, MOE_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    assert r.returncode != 0 and failed, f"mutant {n} ({MUTANTS[n]}) passed every pin"
