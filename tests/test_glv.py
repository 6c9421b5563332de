"""The GLV endomorphism the CUDA path uses to split every scalar in two,
pinned on the CPU: phi(x, y) = (beta x, y) must equal [lambda](x, y) on G1
under the oracle's group law, beta and lambda must be non-trivial cube roots of
unity mod p and mod r, and the split k = k1 + lambda k2 (mod r) must hold with
|k1|, |k2| < 2^127 -- the 128-bit window layout of the GLV path relies on that
bound (Gallant, Lambert, Vanstone, "Faster point multiplication on elliptic
curves with efficient endomorphisms", CRYPTO 2001).

The constants are read from the built library (host-only call, no GPU); the
split is the library's own header compiled for the host.
"""
import os
import random
import subprocess

import numpy as np
import pytest

import oracle
from oracle import pyref
from elliptic_curve_scalar_gb300 import build as lib_build
from elliptic_curve_scalar_gb300 import msm as gm

P, R = pyref.P, pyref.R
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "elliptic_curve_scalar_gb300", "csrc")


@pytest.fixture(scope="module")
def constants():
    lib_build.build()
    beta_mont, lam = gm.glv_constants()
    beta = beta_mont * pow(1 << 256, P - 2, P) % P  # out of Montgomery form
    return beta, lam


def test_cube_roots_of_unity(constants):
    beta, lam = constants
    assert beta not in (0, 1) and (beta * beta + beta + 1) % P == 0
    assert lam not in (0, 1) and (lam * lam + lam + 1) % R == 0


@pytest.mark.parametrize("t", [1, 2, 7, 123456789, R - 1, (R - 1) // 2])
def test_endomorphism_is_multiplication_by_lambda(constants, t):
    """phi([t]G) = [lambda t]G, checked with the C oracle's scalar
    multiplication and, for a few points, the Python affine oracle."""
    beta, lam = constants
    pt = oracle.words_to_point(oracle.generator_multiples(oracle.ints_to_limbs([t]))[0])
    phi = (beta * pt[0] % P, pt[1])
    got = oracle.words_to_point(oracle.scalar_mul(oracle.point_to_words(pt), oracle.int_to_limbs(lam)))
    assert got == phi
    if t < 10:
        assert pyref.mul(lam, pt) == phi


def test_the_other_root_does_not_match(constants):
    """A plausible slip -- pairing beta with lambda^2 instead of lambda -- is
    caught: phi acts as lambda, not as lambda^2."""
    beta, lam = constants
    pt = pyref.mul(5, pyref.G)
    assert pyref.mul(lam * lam % R, pt) != (beta * pt[0] % P, pt[1])


@pytest.fixture(scope="module")
def split_host(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("glv") / "glv_split_host")
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, "-o", exe, os.path.join(ROOT, "tests", "glv_split_host.cpp")],
                   check=True)

    def split(ks):
        text = "\n".join(" ".join("%x" % ((k >> (32 * i)) & 0xFFFFFFFF) for i in range(8)) for k in ks)
        lines = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
        out = []
        for line in lines[:len(ks)]:
            s1, a, s2, b = line.split()
            out.append(((-1 if s1 == "1" else 1) * int(a, 16), (-1 if s2 == "1" else 1) * int(b, 16)))
        return out

    return split


def edge_scalars(lam):
    ks = [0, 1, 2, 3, R - 1, R - 2, lam, R - lam, lam * lam % R, (R - 1) // 2, (R + 1) // 2, 1 << 127, (1 << 128) - 1,
          1 << 128, 1 << 200, (1 << 253) - 1]
    # scalars near the multiples of r / 2^k, where the rounding of x1, x2 is tightest
    ks += [(R * j) >> s for s in (1, 2, 3, 64, 127) for j in (1, 3)]
    return ks


def test_split_identity_and_bound(constants, split_host):
    _, lam = constants
    rng = random.Random(7)
    ks = edge_scalars(lam) + [rng.randrange(R) for _ in range(20000)]
    widest = 0
    for k, (k1, k2) in zip(ks, split_host(ks)):
        assert (k1 + lam * k2 - k) % R == 0, k
        assert abs(k1) < 1 << 127 and abs(k2) < 1 << 127, k
        widest = max(widest, abs(k1).bit_length(), abs(k2).bit_length())
    assert widest >= 125  # the halves really are about half the bits, not trivially small
    assert split_host([0]) == [(0, 0)]
    assert split_host([1]) == [(1, 0)]
