"""The oracle still reproduces the stored small cases (tests/golden/small_msm.json)."""
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "small_msm.json")


def load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_oracle_reproduces_golden(case):
    r = oracle.ints_to_limbs([int(v, 16) for v in case["r"]])
    k = oracle.ints_to_limbs([int(v, 16) for v in case["k"]])
    got = oracle.words_to_point(oracle.msm(oracle.generator_multiples(r, threads=1), k, threads=1))
    expect = None if case["expect"] is None else tuple(int(v, 16) for v in case["expect"])
    assert got == expect
