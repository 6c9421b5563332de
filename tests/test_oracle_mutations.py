"""Plant one mistake at a time in the C oracle (on the CPU) and check that the
pins reject every variant: evidence that the pins pin the oracle."""
import os

import pytest

import oracle
from oracle import build as oracle_build
from tests import oracle_pins

MUTATIONS = {
    1: "doubling drops the -8Y^4 term",
    2: "addition flips the sign of S1*H^3 in Y3",
    3: "Barrett reduction omits the final correction",
    4: "scalar multiplication skips bit 255",
    5: "MSM drops the last term of each thread's range",
    6: "Montgomery decoding multiplies by R instead of R^-1",
    7: "comb table indexed by the wrong byte of the scalar",
    8: "addition of equal points returns infinity instead of doubling",
    9: "the curve-membership test accepts every point",
    10: "the curve-membership test skips its range check on the coordinates",
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return str(tmp_path_factory.mktemp("oracle_mutants"))


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: "M%d" % m)
def test_pins_reject_mutation(mutation, mutant_dir):
    path = os.path.join(mutant_dir, "liboracle_m%d.so" % mutation)
    oracle_build.build(force=True, out=path, mutation=mutation)
    with oracle.use_library(path):
        failed = oracle_pins.failing_pins()
    assert failed, "no pin caught mutation %d (%s)" % (mutation, MUTATIONS[mutation])
