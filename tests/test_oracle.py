"""The CPU oracle against facts fixed by mathematics (see tests/oracle_pins.py)."""
import sympy
import pytest

from oracle import pyref
from tests import oracle_pins


def test_curve_constants():
    """p and r are BN254's from u = 4965661367192848881, both prime, and the
    Montgomery constant the GPU path relies on is -p^-1 mod 2^32."""
    u = 4965661367192848881
    assert pyref.P == 36 * u**4 + 36 * u**3 + 24 * u**2 + 6 * u + 1
    assert pyref.R == 36 * u**4 + 36 * u**3 + 18 * u**2 + 6 * u + 1
    assert hex(pyref.P) == "0x30644e72e131a029b85045b68181585d97816a916871ca8d3c208c16d87cfd47"
    assert hex(pyref.R) == "0x30644e72e131a029b85045b68181585d2833e84879b9709143e1f593f0000001"
    assert sympy.isprime(pyref.P) and sympy.isprime(pyref.R)
    # 3 is not a square mod p, so no curve point has x = 0 and (0, 0) can encode infinity
    assert pow(3, (pyref.P - 1) // 2, pyref.P) == pyref.P - 1
    # the group of points has prime order r (Hasse bound window holds exactly one multiple of r)
    assert abs(pyref.P + 1 - pyref.R) <= 2 * int(sympy.sqrt(pyref.P)) + 2


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


def test_pyref_matches_brute_force_small_multiples():
    """pyref.mul (double and add) agrees with repeated addition for k < 40."""
    p = pyref.mul(31337, pyref.G)
    for k in range(40):
        assert pyref.mul(k, p) == pyref.mul_repeated(k, p)
