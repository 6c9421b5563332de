"""CPU oracle for BN254 G1 multi-scalar multiplication.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``elliptic_curve_scalar_gb300``) never imports it and shares no code with it.

Two independent implementations live here:

* ``msm_oracle.c`` (via ctypes): 4 x 64-bit limbs, canonical residues, Barrett
  reduction, textbook Jacobian double-and-add per term, summed; pthreads over
  terms.  Used for every size.
* ``pyref.py``: Python integers, affine chord-and-tangent law.  Used for tiny
  sizes and to pin the C oracle.

Array conventions (numpy): field elements are ``uint64[..., 4]`` little-endian
limbs; an affine point is ``uint64[8]`` = x[4], y[4]; (0, 0) is infinity.  The
GPU library's ``uint32[..., 8]`` layout is the same bytes on little-endian
hosts, so ``a.view(np.uint64)`` converts.
"""
import ctypes
import os

import numpy as np

from . import build as _build
from . import pyref  # noqa: F401  (re-exported)

_U64P = ctypes.POINTER(ctypes.c_uint64)

_SIGNATURES = [
    ("oracle_init", []),
    ("oracle_g1_generator_multiples", [_U64P, ctypes.c_size_t, _U64P, ctypes.c_int]),
    ("oracle_msm", [_U64P, _U64P, ctypes.c_size_t, _U64P, ctypes.c_int]),
    ("oracle_mont_encode", [_U64P, ctypes.c_size_t, _U64P]),
    ("oracle_mont_decode", [_U64P, ctypes.c_size_t, _U64P]),
    ("oracle_jacobian_mont_to_affine", [_U64P, _U64P]),
    ("oracle_g1_add", [_U64P, _U64P, _U64P]),
    ("oracle_g1_scalar_mul", [_U64P, _U64P, _U64P]),
    ("oracle_g1_is_on_curve", [_U64P]),
    ("oracle_scalar_dot_mod_r", [_U64P, _U64P, ctypes.c_size_t, _U64P]),
    ("oracle_fp_mul", [_U64P, _U64P, _U64P]),
    ("oracle_fp_inv", [_U64P, _U64P]),
]

_libs = {}


def load_library(path=None):
    """ctypes handle on a built oracle (the default build unless ``path`` is given)."""
    path = path or _build.build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        for name, args in _SIGNATURES:
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.oracle_init()
        _libs[path] = lib
    return _libs[path]


_active = [None]


def _load():
    if _active[0] is None:
        _active[0] = load_library()
    return _active[0]


class use_library:
    """Context manager that routes this module's functions to another build
    (used by the mutation tests to run the pins against a planted mistake)."""

    def __init__(self, path):
        self.lib = load_library(path)

    def __enter__(self):
        self.prev = _active[0]
        _active[0] = self.lib
        return self.lib

    def __exit__(self, *exc):
        _active[0] = self.prev
        return False


def default_threads():
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _u64(a, shape_tail):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.uint64)
    a = np.ascontiguousarray(a, dtype=np.uint64)
    return a.reshape((-1,) + shape_tail)


def _ptr(a):
    return a.ctypes.data_as(_U64P)


# ------------------------------------------------------------ int <-> limbs

def int_to_limbs(x, nlimbs=4):
    return np.array([(x >> (64 * i)) & 0xFFFFFFFFFFFFFFFF for i in range(nlimbs)], dtype=np.uint64)


def limbs_to_int(a):
    a = np.asarray(a, dtype=np.uint64).reshape(-1)
    return sum(int(v) << (64 * i) for i, v in enumerate(a))


def ints_to_limbs(xs):
    out = np.zeros((len(xs), 4), dtype=np.uint64)
    for i, x in enumerate(xs):
        out[i] = int_to_limbs(x)
    return out


def point_to_words(pt):
    """pyref point (tuple or None) -> uint64[8]"""
    if pt is None:
        return np.zeros(8, dtype=np.uint64)
    return np.concatenate([int_to_limbs(pt[0]), int_to_limbs(pt[1])])


def words_to_point(w):
    w = np.asarray(w, dtype=np.uint64).reshape(8)
    x, y = limbs_to_int(w[:4]), limbs_to_int(w[4:])
    if x == 0 and y == 0:
        return None
    return (x, y)


# ------------------------------------------------------------------ oracle

def generator_multiples(k, threads=None):
    """uint64[n, 4] scalars -> uint64[n, 8] canonical affine points [k_i]G."""
    k = _u64(k, (4,))
    out = np.zeros((k.shape[0], 8), dtype=np.uint64)
    rc = _load().oracle_g1_generator_multiples(_ptr(k), k.shape[0], _ptr(out), threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_g1_generator_multiples failed")
    return out


def msm(points_affine, scalars, threads=None):
    """canonical affine uint64[n, 8], scalars uint64[n, 4] -> canonical affine uint64[8]."""
    pts = _u64(points_affine, (8,))
    k = _u64(scalars, (4,))
    if pts.shape[0] != k.shape[0]:
        raise ValueError("points and scalars differ in length")
    out = np.zeros(8, dtype=np.uint64)
    rc = _load().oracle_msm(_ptr(pts), _ptr(k), pts.shape[0], _ptr(out), threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_msm failed")
    return out


def mont_encode(a):
    """canonical field elements (uint64[..., 4]) -> Montgomery form x * 2^256 mod p."""
    a = np.asarray(a)
    shape = a.shape if a.dtype == np.uint64 else a.view(np.uint64).shape
    flat = _u64(a, (4,))
    out = np.zeros_like(flat)
    _load().oracle_mont_encode(_ptr(flat), flat.shape[0], _ptr(out))
    return out.reshape(shape)


def mont_decode(a):
    a = np.asarray(a)
    shape = a.shape if a.dtype == np.uint64 else a.view(np.uint64).shape
    flat = _u64(a, (4,))
    out = np.zeros_like(flat)
    _load().oracle_mont_decode(_ptr(flat), flat.shape[0], _ptr(out))
    return out.reshape(shape)


def points_to_gpu_layout(points_affine):
    """canonical affine uint64[n, 8] -> Montgomery affine uint32[n, 16] (the GPU input layout)."""
    pts = _u64(points_affine, (8,))
    enc = mont_encode(pts.reshape(-1, 4)).reshape(-1, 8)
    inf = np.all(pts == 0, axis=1)
    enc[inf] = 0  # (0, 0) encodes infinity in both layouts
    return np.ascontiguousarray(enc).view(np.uint32).reshape(-1, 16)


def jacobian_mont_to_affine(jac):
    """GPU output (uint32[24] or uint64[12], Montgomery X, Y, Z) -> canonical affine uint64[8]."""
    j = _u64(jac, (12,)).reshape(12)
    out = np.zeros(8, dtype=np.uint64)
    _load().oracle_jacobian_mont_to_affine(_ptr(j), _ptr(out))
    return out


def add(a, b):
    a, b = _u64(a, (8,)).reshape(8), _u64(b, (8,)).reshape(8)
    out = np.zeros(8, dtype=np.uint64)
    _load().oracle_g1_add(_ptr(a), _ptr(b), _ptr(out))
    return out


def scalar_mul(pt, k):
    pt = _u64(pt, (8,)).reshape(8)
    k = _u64(k, (4,)).reshape(4)
    out = np.zeros(8, dtype=np.uint64)
    _load().oracle_g1_scalar_mul(_ptr(pt), _ptr(k), _ptr(out))
    return out


def is_on_curve(pt):
    pt = _u64(pt, (8,)).reshape(8)
    return bool(_load().oracle_g1_is_on_curve(_ptr(pt)))


def scalar_dot_mod_r(a, b):
    a, b = _u64(a, (4,)), _u64(b, (4,))
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_scalar_dot_mod_r(_ptr(a), _ptr(b), a.shape[0], _ptr(out))
    return out


def fp_mul(a, b):
    a, b = _u64(a, (4,)).reshape(4), _u64(b, (4,)).reshape(4)
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_fp_mul(_ptr(a), _ptr(b), _ptr(out))
    return out


def fp_inv(a):
    a = _u64(a, (4,)).reshape(4)
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_fp_inv(_ptr(a), _ptr(out))
    return out


def closed_form(r_values, scalars):
    """For points P_i = [r_i]G: sum_i k_i P_i = [sum_i k_i r_i mod r]G."""
    s = scalar_dot_mod_r(r_values, scalars)
    return generator_multiples(s.reshape(1, 4), threads=1)[0]
