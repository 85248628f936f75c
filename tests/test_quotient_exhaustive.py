"""The indexer-K store kernel replaces the rule's per-element IEEE division
k / scale by an FMA-corrected product (q0 = k * RN(1/scale), one residual
r = k - q0 * scale, q1 = q0 + r * RN(1/scale), the sign bit of k OR-ed into
the code).  ``quotient_exhaustive.c`` enumerates every pair (amax, k) of
finite bf16 or fp16 inputs with |k| <= amax and amax / 448 >= 2^-90 (the
kernel's fast-path condition) and counts the pairs whose e4m3 code could
differ from that of the IEEE quotient.  CPU only; the enumeration also
shows mismatches for the uncorrected product, so it can fail."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "quotient_exhaustive.c")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("qex") / "quotient_exhaustive")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-pthread", SRC, "-o",
                    exe, "-lm"], check=True)
    return exe


def _run(exe, kind, *extra):
    threads = str(max(1, min(os.cpu_count() or 1, 32)))
    out = subprocess.run([exe, kind, threads, *extra], check=True,
                         capture_output=True, text=True).stdout.split()
    assert out[0] == kind
    return int(out[1]), int(out[2])


@pytest.mark.parametrize("kind", ["bf16", "fp16"])
def test_corrected_quotient_gives_the_ieee_code_for_every_pair(checker, kind):
    pairs, bad = _run(checker, kind)
    assert pairs > 10 ** 9          # both signs of every |k| <= amax
    assert bad == 0


def test_the_enumeration_detects_an_uncorrected_product(checker):
    pairs, bad = _run(checker, "fp16", "uncorrected")
    assert pairs > 10 ** 9 and bad > 10 ** 6
