"""Write tests/golden/small_msm.json: small seeded MSM cases with expected results.

The pages print no worked example with values, so every expected value here is
computed by the CPU oracle (``oracle.msm``) and, before it is written, checked
against the independent pure-Python oracle (``oracle.pyref``).  Only ``oracle/``
and the seeded workload generator are called.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import pyref  # noqa: E402
from elliptic_curve_scalar_gb300 import synth  # noqa: E402


def case(name, r_ints, k_ints):
    r_l = oracle.ints_to_limbs(r_ints)
    k_l = oracle.ints_to_limbs(k_ints)
    pts = oracle.generator_multiples(r_l, threads=2)
    got = oracle.words_to_point(oracle.msm(pts, k_l, threads=2))
    expect = pyref.msm([pyref.mul(r, pyref.G) for r in r_ints], k_ints)
    assert got == expect, name
    return {
        "name": name,
        "r": [hex(v) for v in r_ints],
        "k": [hex(v) for v in k_ints],
        "expect": None if got is None else [hex(got[0]), hex(got[1])],
    }


def main():
    R = pyref.R
    cases = []
    r, k = synth.uniform_workload(8, 1)
    cases.append(case("uniform_n8_seed1", synth.limbs_to_ints(r), synth.limbs_to_ints(k)))
    r, k = synth.progression_workload(12, 3, scalars="ones")
    cases.append(case("progression_ones_n12", synth.limbs_to_ints(r), synth.limbs_to_ints(k)))
    a, b = 123456789, 987654321
    cases.append(case("dup_and_neg", [a, a, R - a, b], [5, 7, 2, 1]))
    cases.append(case("single_r_minus_1", [a], [R - 1]))
    cases.append(case("all_zero", [a, b], [0, 0]))
    cases.append(case("cancel_to_infinity", [a, R - a], [3, 3]))
    cases.append(case("large_scalars", [a, b], [(1 << 256) - 1, R]))
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "small_msm.json")
    with open(out, "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (oracle.msm, cross-checked with oracle.pyref)",
                   "curve": "BN254 G1, y^2 = x^3 + 3, G = (1, 2)",
                   "points": "P_i = [r_i]G", "cases": cases}, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
