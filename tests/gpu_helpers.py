"""Shared helpers for the GPU parity tests.

Inputs always come from the seeded generator (elliptic_curve_scalar_gb300.synth)
and the CPU oracle (points P_i = [r_i]G computed by oracle.generator_multiples);
expected values always come from the oracle.  Results of the CUDA path are
normalised to canonical affine coordinates by the oracle before comparing.
"""
import numpy as np
import torch

import oracle
from oracle import pyref
from elliptic_curve_scalar_gb300 import msm as gm
from elliptic_curve_scalar_gb300 import synth

P, R = pyref.P, pyref.R
RMONT = (1 << 256) % P


def mont(x):
    return x * RMONT % P


def unmont(x):
    return x * pow(RMONT, P - 2, P) % P


def ints_to_u32(xs):
    """python ints -> uint32[n, 8]"""
    out = np.zeros((len(xs), 8), dtype=np.uint32)
    for i, x in enumerate(xs):
        for j in range(8):
            out[i, j] = (x >> (32 * j)) & 0xFFFFFFFF
    return out


def u32_to_ints(a):
    a = np.asarray(a, dtype=np.uint32).reshape(-1, 8)
    return [sum(int(v) << (32 * j) for j, v in enumerate(row)) for row in a]


def points_from_r(r_values):
    """oracle: r_i -> canonical affine uint64[n, 8]"""
    return oracle.generator_multiples(r_values)


def gpu_points(points_affine):
    """canonical affine (uint64[n, 8]) -> device tensor in the library layout"""
    return gm.to_device(oracle.points_to_gpu_layout(points_affine))


def gpu_scalars(k):
    return gm.to_device(synth.scalars_to_u32(k))


def normalise(out_tensor):
    """GPU Jacobian result -> canonical affine uint64[8] via the oracle"""
    torch.cuda.synchronize()
    return oracle.jacobian_mont_to_affine(gm.to_host(out_tensor))


def aff_words_to_point(words_u32):
    """(16,) uint32 Montgomery affine -> pyref point"""
    w = np.asarray(words_u32, dtype=np.uint32)
    x, y = u32_to_ints(w[:8])[0], u32_to_ints(w[8:16])[0]
    if x == 0 and y == 0:
        return None
    return (unmont(x), unmont(y))


def point_to_aff_words(pt):
    if pt is None:
        return np.zeros(16, dtype=np.uint32)
    return np.concatenate([ints_to_u32([mont(pt[0])])[0], ints_to_u32([mont(pt[1])])[0]])


def point_to_jac_words(pt, z=1):
    """pyref point -> (24,) uint32 Montgomery Jacobian with the given Z"""
    if pt is None:
        return np.concatenate([ints_to_u32([mont(1), mont(1), 0]).reshape(-1)])
    X, Y, Z = pt[0] * z * z % P, pt[1] * z * z * z % P, z % P
    return ints_to_u32([mont(X), mont(Y), mont(Z)]).reshape(-1)


def jac_words_to_point(w):
    X, Y, Z = (unmont(v) for v in u32_to_ints(np.asarray(w, dtype=np.uint32).reshape(3, 8)))
    if Z == 0:
        return None
    zi = pow(Z, P - 2, P)
    return (X * zi * zi % P, Y * zi * zi * zi % P)
