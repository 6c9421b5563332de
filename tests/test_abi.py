"""The C-ABI library loads, exports every function include/*.h declares, and
its host-side logic (argument checks, sizing helpers) works without a GPU."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from elliptic_curve_scalar_gb300 import build as lib_build
from elliptic_curve_scalar_gb300 import msm as gm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(msm_g1_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return gm.lib()


def test_headers_declare_the_boundary():
    names = declared_functions()
    for must in ("msm_g1_create", "msm_g1_run", "msm_g1_destroy"):
        assert must in names
    assert len(names) >= 15


@pytest.mark.parametrize("name", declared_functions())
def test_symbol_exported(lib, name):
    assert hasattr(lib, name), name


def _cuda_include():
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.exists(os.path.join(base, "include", "cuda_runtime_api.h")):
            return os.path.join(base, "include")
    return None


def test_headers_compile_and_link_as_c(lib, tmp_path):
    """The boundary is plain C: the headers compile as C11 (warnings as errors)
    and a C program links against the library, resolving every declared entry
    point, then runs the host-only helpers."""
    gcc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if not gcc or not inc:
        pytest.skip("no C compiler or CUDA headers")
    src = os.path.join(ROOT, "tests", "c_abi_check.c")
    text = open(src).read()
    for name in declared_functions():
        assert "(any_fn)%s," % name in text, name
    libdir = os.path.dirname(lib_build.LIB)
    exe = str(tmp_path / "c_abi_check")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-isystem", inc, src, "-o", exe, "-L", libdir, "-lmsm_g1", "-Wl,-rpath," + libdir]
    built = subprocess.run(cmd, capture_output=True, text=True)
    assert built.returncode == 0, built.stdout + built.stderr
    ran = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert ran.returncode == 0 and "c abi ok" in ran.stdout, (ran.returncode, ran.stdout, ran.stderr)


def test_window_count(lib):
    for c in range(1, 21):
        assert lib.msm_g1_window_count(c) == -(-255 // c)
    assert lib.msm_g1_window_count(0) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_window_count(21) == gm.ERR_INVALID_ARG


def test_auto_window(lib):
    assert lib.msm_g1_auto_window(1 << 10) == 8
    assert lib.msm_g1_auto_window(1 << 16) == 13
    assert lib.msm_g1_auto_window(1 << 20) == 16
    for n in (1, 2, 1000, 1 << 30):
        assert 4 <= lib.msm_g1_auto_window(n) <= 18


def test_scratch_bytes(lib):
    a = lib.msm_g1_scratch_bytes(1 << 16, 13)
    b = lib.msm_g1_scratch_bytes(1 << 20, 13)
    c = lib.msm_g1_scratch_bytes(1 << 20, 16)
    assert 0 < a < b <= c
    # entries (4 B) and level-1 items (32 B per entry) dominate: n * W(8) * 36 B
    assert b >= (1 << 20) * 32 * 36
    assert lib.msm_g1_scratch_bytes(0, 8) == 0
    assert lib.msm_g1_scratch_bytes(16, 0) == 0


def test_noalloc_scratch_holds_its_documented_limit(lib):
    """msm_g1_run_noalloc serves n <= 4096, c <= 10 from a fixed 8 MiB device
    array; the sizing of a context for that limit must fit in it (a change of
    the buffers' sizes that breaks this would make every such call fail)."""
    assert 0 < lib.msm_g1_scratch_bytes(4096, 10) <= 8 << 20


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert lib.msm_g1_strerror(code)


def test_argument_checks_before_device_work(lib):
    """Null contexts and bad sizes are rejected on the host."""
    vp = ctypes.c_void_p
    assert lib.msm_g1_create(None, 16, 8) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_create_batch(None, 16, 8, 4) == gm.ERR_INVALID_ARG
    ctx = vp()
    assert lib.msm_g1_create(ctypes.byref(ctx), 16, 0) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_create(ctypes.byref(ctx), 0, 8) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_create(ctypes.byref(ctx), 16, 21) == gm.ERR_INVALID_ARG
    assert not ctx.value
    assert lib.msm_g1_run(None, None, None, 0, 8, None, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_run_host(None, None, None, 0, 8, None, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_run_batch(None, None, None, None, 1, 8, None, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_set_param(None, gm.PARAM_BATCH_S, 8) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_mul_generator(None, None, 0, None, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_test_fq(99, None, None, None, 1, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_test_batch_add(vp(16), vp(16), vp(16), 4, 3, 0, None) == gm.ERR_INVALID_ARG
    assert lib.msm_g1_test_batch_add(vp(16), vp(16), vp(16), 4, 4, 4, None) == gm.ERR_INVALID_ARG
    lib.msm_g1_destroy(None)


def test_no_device_is_reported():
    """Without a GB300 the library refuses to create a context (no CPU path)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ctx = ctypes.c_void_p()
    rc = gm.lib().msm_g1_create(ctypes.byref(ctx), 16, 8)
    assert rc == gm.ERR_NO_DEVICE and not ctx.value
    with pytest.raises(gm.MsmError):
        gm.MsmG1(16, 8)
