"""Thin ctypes binding of libmsm_g1.so (the C ABI in include/msm_g1.h).

Argument marshalling only: every step of the MSM runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is not built, or no GB300 is present, calls raise.

Tensor conventions (all on the same CUDA device, contiguous, torch.int32
holding the uint32 words bit for bit):
  points  (n, 16)  affine x[8], y[8], Montgomery form, (0, 0) = infinity
  scalars (n, 8)   plain little-endian integers < 2^256
  result  (24,)    Jacobian X[8], Y[8], Z[8], Montgomery form, Z = 0 = infinity
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = -1
ERR_CUDA = -2
ERR_CAPACITY = -3
ERR_ALLOC = -4
ERR_NO_DEVICE = -5
MAX_WINDOW = 20

PARAM_BATCH_S = 1
PARAM_TPB = 2
PARAM_TIMING = 3
PARAM_STATS = 4
PARAM_GROUPS = 5
PARAM_FINISH = 6
PARAM_GLV = 7
PARAM_INVERSION = 8
PARAM_GRAPH = 9
PARAM_GRID = 10
PARAM_ACC_PLACEMENT = 11
ACC_LOCAL = 0
ACC_SHARED = 1
ACC_REGISTERS = 2
PLAIN_BITS = 255  # bits the signed windows of a scalar mod r cover
GLV_BITS = 128    # bits the signed windows of one GLV half cover

PHASES = ("digits", "scan", "scatter", "accum_l0", "accum_tree", "bucket_reduce", "combine")
STATS = ("entries", "nonempty_buckets", "max_bucket", "adds", "inversions", "levels", "launches", "error",
         "finish_t", "chunk_len", "groups")

TEST_FQ = {"mul": 0, "sqr": 1, "add": 2, "sub": 3, "neg": 4, "inv": 5, "inv_fermat": 6, "inv_table": 7, "inv_block": 8}
TEST_G1 = {"jac_dbl": 0, "jac_add": 1, "jac_mixed": 2, "to_affine": 3, "jac_dbl_coop": 4, "jac_add_coop": 5,
           "jac_mixed_coop": 6, "jac_dbl_coop8": 7, "jac_add_coop8": 8, "jac_mixed_coop8": 9, "jac_dbl5_coop": 10,
           "aff_add": 11}

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int

_SIGS = {
    "msm_g1_create": (_i, [ctypes.POINTER(_vp), _sz, _i]),
    "msm_g1_create_batch": (_i, [ctypes.POINTER(_vp), _sz, _i, _i]),
    "msm_g1_run": (_i, [_vp, _vp, _vp, _sz, _i, _vp, _vp]),
    "msm_g1_run_noalloc": (_i, [_vp, _vp, _sz, _i, _vp, _vp]),
    "msm_g1_run_host": (_i, [_vp, _vp, _vp, _sz, _i, _vp, _vp]),
    "msm_g1_run_batch": (_i, [_vp, _vp, _vp, ctypes.POINTER(_sz), _i, _i, _vp, _vp]),
    "msm_g1_mul_generator": (_i, [_vp, _vp, _sz, _vp, _vp]),
    "msm_g1_destroy": (None, [_vp]),
    "msm_g1_set_param": (_i, [_vp, _i, _i]),
    "msm_g1_get_param": (_i, [_vp, _i, ctypes.POINTER(_i)]),
    "msm_g1_last_phase_ms": (_i, [_vp, ctypes.POINTER(ctypes.c_float), _i]),
    "msm_g1_last_stats": (_i, [_vp, ctypes.POINTER(ctypes.c_uint64), _i]),
    "msm_g1_window_count": (_i, [_i]),
    "msm_g1_auto_window": (_i, [_sz]),
    "msm_g1_scratch_bytes": (_sz, [_sz, _i]),
    "msm_g1_strerror": (ctypes.c_char_p, [_i]),
    "msm_g1_test_fq": (_i, [_i, _vp, _vp, _vp, _sz, _vp]),
    "msm_g1_test_g1": (_i, [_i, _vp, _vp, _vp, _sz, _vp]),
    "msm_g1_test_batch_add": (_i, [_vp, _vp, _vp, _sz, _i, _i, _vp]),
    "msm_g1_test_digits": (_i, [_vp, _sz, _i, _i, _vp, _vp]),
    "msm_g1_test_glv_split": (_i, [_vp, _sz, _vp, _vp]),
    "msm_g1_test_rns": (_i, [_i, _vp, _vp, _vp, _sz, _i, _vp]),
    "msm_g1_glv_constants": (_i, [_vp, _vp]),
    "msm_g1_debug_read": (_i, [_vp, _i, _vp, _sz, ctypes.POINTER(_sz)]),
}

_lib = None


def library_path():
    return _build.LIB


def lib():
    """The loaded libmsm_g1.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libmsm_g1.so is not built (%s); run elliptic_curve_scalar_gb300.build.build()" % path)
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class MsmError(RuntimeError):
    def __init__(self, code, what):
        msg = lib().msm_g1_strerror(code).decode()
        super().__init__("%s failed: %s (%d)" % (what, msg, code))
        self.code = code


def _check(code, what):
    if code != OK:
        raise MsmError(code, what)
    return code


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_u32(t, shape_tail, what):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous torch.int32 tensor" % what)
    if tuple(t.shape[1:]) != shape_tail:
        raise ValueError("%s must have shape (n,) + %s" % (what, shape_tail))
    return ctypes.c_void_p(t.data_ptr())


def to_device(a, device="cuda"):
    """numpy uint32/uint64 words -> CUDA int32 tensor (same bytes)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint64:
        a = a.view(np.uint32).reshape(a.shape[:-1] + (a.shape[-1] * 2,))
    return torch.from_numpy(a.view(np.int32)).to(device)


def to_host(t):
    """CUDA int32 tensor -> numpy uint32 (same bytes)."""
    return t.detach().cpu().numpy().view(np.uint32)


def window_count(c):
    return lib().msm_g1_window_count(c)


def auto_window(n):
    return lib().msm_g1_auto_window(n)


def scratch_bytes(max_n, max_c):
    return lib().msm_g1_scratch_bytes(max_n, max_c)


class MsmG1:
    """One MSM context: device scratch for n <= max_n and c <= max_c."""

    def __init__(self, max_n, max_c=16, device=None, max_batch=1):
        self._ctx = ctypes.c_void_p()
        if not torch.cuda.is_available():
            raise MsmError(ERR_NO_DEVICE, "msm_g1_create")
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        with torch.cuda.device(self.device):
            _check(lib().msm_g1_create_batch(ctypes.byref(self._ctx), max_n, max_c, max_batch),
                   "msm_g1_create_batch")
        self.max_n = max_n
        self.max_c = max_c

    def close(self):
        if self._ctx:
            lib().msm_g1_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def set_param(self, key, value):
        _check(lib().msm_g1_set_param(self._ctx, key, value), "msm_g1_set_param")

    def get_param(self, key):
        v = ctypes.c_int()
        _check(lib().msm_g1_get_param(self._ctx, key, ctypes.byref(v)), "msm_g1_get_param")
        return v.value

    def run(self, points, scalars, c=0, out=None, stream=None):
        """Q = sum_i k_i P_i as a (24,) int32 Jacobian tensor (asynchronous)."""
        n = scalars.shape[0]
        if points.shape[0] != n:
            raise ValueError("points and scalars differ in length")
        pp = _dev_u32(points, (16,), "points")
        sp = _dev_u32(scalars, (8,), "scalars")
        if out is None:
            out = torch.empty(24, dtype=torch.int32, device=points.device)
        op = ctypes.c_void_p(out.data_ptr())
        with torch.cuda.device(self.device):
            _check(lib().msm_g1_run(self._ctx, pp, sp, n, c, op, _stream_handle(stream)), "msm_g1_run")
        return out

    def run_batch(self, points, scalars, offsets, c=0, out=None, stream=None):
        """msm_g1_run_batch: len(offsets) - 1 MSMs over the concatenated terms;
        returns a (count, 24) int32 tensor of Jacobian results (asynchronous)."""
        count = len(offsets) - 1
        if count < 1 or points.shape[0] != scalars.shape[0] or offsets[-1] != scalars.shape[0]:
            raise ValueError("offsets must span the concatenated terms")
        pp = _dev_u32(points, (16,), "points")
        sp = _dev_u32(scalars, (8,), "scalars")
        if out is None:
            out = torch.empty((count, 24), dtype=torch.int32, device=points.device)
        offs = (ctypes.c_size_t * (count + 1))(*[int(o) for o in offsets])
        with torch.cuda.device(self.device):
            _check(lib().msm_g1_run_batch(self._ctx, pp, sp, offs, count, c, ctypes.c_void_p(out.data_ptr()),
                                          _stream_handle(stream)), "msm_g1_run_batch")
        return out

    def run_host(self, points, scalars, c=0, out=None, stream=None):
        """msm_g1_run_host: inputs and result in host memory (CPU torch tensors,
        pinned for asynchronous copies).  Returns the (24,) int32 CPU result
        tensor, valid once the stream has been synchronised."""
        n = scalars.shape[0]
        if points.shape[0] != n:
            raise ValueError("points and scalars differ in length")
        for t, tail, what in ((points, (16,), "points"), (scalars, (8,), "scalars")):
            if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous() \
                    or tuple(t.shape[1:]) != tail:
                raise TypeError("%s must be a contiguous CPU torch.int32 tensor of shape (n,) + %s" % (what, tail))
        if out is None:
            out = torch.empty(24, dtype=torch.int32).pin_memory()
        with torch.cuda.device(self.device):
            _check(lib().msm_g1_run_host(self._ctx, ctypes.c_void_p(points.data_ptr()),
                                         ctypes.c_void_p(scalars.data_ptr()), n, c, ctypes.c_void_p(out.data_ptr()),
                                         _stream_handle(stream)), "msm_g1_run_host")
        return out

    def mul_generator(self, scalars, out=None, stream=None):
        """[k_i]G for each scalar, (n, 16) int32 affine Montgomery points."""
        n = scalars.shape[0]
        sp = _dev_u32(scalars, (8,), "scalars")
        if out is None:
            out = torch.empty((n, 16), dtype=torch.int32, device=scalars.device)
        with torch.cuda.device(self.device):
            _check(lib().msm_g1_mul_generator(self._ctx, sp, n, ctypes.c_void_p(out.data_ptr()),
                                              _stream_handle(stream)), "msm_g1_mul_generator")
        return out

    def phase_ms(self):
        buf = (ctypes.c_float * len(PHASES))()
        k = lib().msm_g1_last_phase_ms(self._ctx, buf, len(PHASES))
        if k < 0:
            raise MsmError(k, "msm_g1_last_phase_ms")
        return dict(zip(PHASES[:k], buf[:k]))

    def stats(self):
        buf = (ctypes.c_uint64 * len(STATS))()
        k = lib().msm_g1_last_stats(self._ctx, buf, len(STATS))
        if k < 0:
            raise MsmError(k, "msm_g1_last_stats")
        return dict(zip(STATS[:k], buf[:k]))

    def debug_read(self, which, nwords):
        """Synchronous copy of an internal buffer of the last run (uint32 words)."""
        out = np.zeros(nwords, dtype=np.uint32)
        nbytes = ctypes.c_size_t()
        _check(lib().msm_g1_debug_read(self._ctx, which, out.ctypes.data_as(ctypes.c_void_p), out.nbytes,
                                       ctypes.byref(nbytes)), "msm_g1_debug_read")
        return out, nbytes.value


def run_noalloc(points, scalars, c=0, out=None, stream=None):
    """msm_g1_run_noalloc: the MSM without a context, for n <= 4096 and c <= 10,
    using the library's fixed device scratch array (see include/msm_g1.h)."""
    n = scalars.shape[0]
    if points.shape[0] != n:
        raise ValueError("points and scalars differ in length")
    pp = _dev_u32(points, (16,), "points")
    sp = _dev_u32(scalars, (8,), "scalars")
    if out is None:
        out = torch.empty(24, dtype=torch.int32, device=points.device)
    _check(lib().msm_g1_run_noalloc(pp, sp, n, c, ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)),
           "msm_g1_run_noalloc")
    return out


# ----------------------------------------------------------------- test hooks

def test_fq(op, a, b=None, stream=None):
    n = a.shape[0]
    out = torch.empty_like(a)
    bp = ctypes.c_void_p(b.data_ptr()) if b is not None else ctypes.c_void_p()
    _check(lib().msm_g1_test_fq(TEST_FQ[op], ctypes.c_void_p(a.data_ptr()), bp, ctypes.c_void_p(out.data_ptr()), n,
                                _stream_handle(stream)), "msm_g1_test_fq")
    return out


def test_g1(op, a, b=None, stream=None):
    n = a.shape[0]
    width = 16 if op == "to_affine" else 24
    out = torch.empty((n, width), dtype=torch.int32, device=a.device)
    bp = ctypes.c_void_p(b.data_ptr()) if b is not None else ctypes.c_void_p()
    _check(lib().msm_g1_test_g1(TEST_G1[op], ctypes.c_void_p(a.data_ptr()), bp, ctypes.c_void_p(out.data_ptr()), n,
                                _stream_handle(stream)), "msm_g1_test_g1")
    return out


def test_batch_add(a, b, batch_s, inline_back=0, block=0, stream=None):
    n = a.shape[0]
    out = torch.empty_like(a)
    mode = (1 if inline_back else 0) | (2 if block else 0)
    _check(lib().msm_g1_test_batch_add(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                       ctypes.c_void_p(out.data_ptr()), n, batch_s, mode,
                                       _stream_handle(stream)),
           "msm_g1_test_batch_add")
    return out


def test_digits(scalars, c, nbits=PLAIN_BITS, stream=None):
    n = scalars.shape[0]
    out = torch.empty((n, -(-nbits // c)), dtype=torch.int32, device=scalars.device)
    _check(lib().msm_g1_test_digits(ctypes.c_void_p(scalars.data_ptr()), n, c, nbits,
                                    ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)), "msm_g1_test_digits")
    return out


def test_glv_split(scalars, stream=None):
    """(n, 10) uint32 words per scalar: |k1| (4), |k2| (4), sign of k1, sign of k2."""
    n = scalars.shape[0]
    out = torch.empty((n, 10), dtype=torch.int32, device=scalars.device)
    _check(lib().msm_g1_test_glv_split(ctypes.c_void_p(scalars.data_ptr()), n, ctypes.c_void_p(out.data_ptr()),
                                       _stream_handle(stream)), "msm_g1_test_glv_split")
    return out


def glv_constants():
    """(beta in Montgomery form, lambda) as Python ints, read from the library
    (host only)."""
    beta = (ctypes.c_uint32 * 8)()
    lam = (ctypes.c_uint32 * 8)()
    _check(lib().msm_g1_glv_constants(beta, lam), "msm_g1_glv_constants")
    return (sum(int(v) << (32 * j) for j, v in enumerate(beta)), sum(int(v) << (32 * j) for j, v in enumerate(lam)))
