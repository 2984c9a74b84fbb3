"""The quantizers' fast quotient equals IEEE division on every BF16 input.

The quantizer kernels form fl32(x / s) with one reciprocal per tile and
Markstein's correction step on negated quantities (see quotient_check.c for
the exact sequence of operations), switching to IEEE division for tiles whose
amax is below 2^-80.  Correct rounding of the quotient is part of the
quantization rule, so that replacement must give the same E4M3 code as IEEE
division for every element the kernels can meet with BF16 input.  These tests
run the check over all pairs of BF16 values (x, amax), |x| <= amax, on the
host CPU (plain C, no GPU).
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "quotient_check.c")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    exe = str(tmp_path_factory.mktemp("qc") / "quotient_check")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-o", exe, SRC, "-lm"],
                   check=True)
    return exe


def run(exe, *args):
    p = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=600)
    checked, failed = (int(t) for t in p.stdout.split()[1::2])
    return p.returncode, checked, failed


def test_every_bf16_pair_matches_ieee_division(checker):
    rc, checked, failed = run(checker)
    # 32,640 finite non-negative BF16 magnitudes; pairs with |x| <= amax,
    # amax >= 2^-80, both signs of x: over 10^9 quotients
    assert checked > 1_000_000_000
    assert failed == 0 and rc == 0


def test_cutoff_is_needed(checker):
    # Without the IEEE fallback for tiny tiles the correction step is not
    # always exact (the residual underflows): the check must see failures,
    # otherwise it could not catch a wrong cutoff either.
    rc, checked, failed = run(checker, 1, -100)
    assert failed > 0 and rc == 1
