"""Planted mistakes in the CUDA path must fail the GPU parity checks.

"Context Parallelism for Long-Context Training", section "Prove attention
equivalence", names the failure to provoke on purpose: a position or mask
seam that is wrong.  Each mutant below is the library compiled with one
planted mistake (CPATTN_MUTATION, csrc/cpattn_internal.h) into a build
folder of its own; tests/mutant_check.py runs the same small parity checks
against the oracle in a separate process, once on the regular library
(every check passes) and once per mutant (the checks named here fail).
The mistakes sit in index or mask arithmetic only, never in a barrier or a
wait, so a mutant computes wrong numbers and cannot hang or fault:

1. the forward's element mask drops the diagonal (the seam between a query
   and its own key);
2. the ring turns the other way (step t brings rank (r + t) mod cp): the
   whole result is unchanged, but the per-step partials and the contiguous
   layout's per-step census are not;
3. the LSE merge drops the second partial's term;
4. the dK / dV kernel forms dS without Delta.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from context_causal_attention_zigzag_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CHECKER = os.path.join(HERE, "mutant_check.py")
MUTANTS = {1: ("forward mask drops the diagonal", {"forward", "step_partials"}),
           2: ("ring turned the other way", {"step_partials", "census"}),
           3: ("LSE merge drops a term", {"merge"}),
           4: ("dS formed without Delta", {"backward"})}


def run_checks(lib):
    p = subprocess.run([sys.executable, CHECKER, lib], capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    return json.loads(p.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def mutant_libs():
    with ThreadPoolExecutor(max_workers=len(MUTANTS)) as ex:
        paths = list(ex.map(lambda m: cuda_build.build(mutation=m), sorted(MUTANTS)))
    return dict(zip(sorted(MUTANTS), paths))


def test_regular_library_passes_every_check():
    res = run_checks(cuda_build.build())
    assert all(res[name] for name in ("forward", "step_partials", "merge", "census",
                                      "backward")), res
    assert res["device_status"] == 0


@pytest.mark.parametrize("m", sorted(MUTANTS), ids=[MUTANTS[m][0] for m in sorted(MUTANTS)])
def test_planted_mistake_is_caught(m, mutant_libs):
    res = run_checks(mutant_libs[m])
    failed = {name for name in ("forward", "step_partials", "merge", "census", "backward")
              if not res[name]}
    assert MUTANTS[m][1] <= failed, (m, res)
