"""Compile the CUDA library (libmsm_g1.so) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into a
shared library next to this file (``_lib/libmsm_g1.so``).  ``ptxas -v``
register and spill figures go to ``_lib/ptxas.log``.
"""
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libmsm_g1.so")
SOURCES = ["msm_g1.cu", "msm_accum.cu", "msm_testing.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force=False, verbose=False):
    """Build libmsm_g1.so if any source is newer; return its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    flags = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
             "-I", INCLUDE] + ARCH
    tmp = tempfile.mkdtemp(prefix="msm_build_", dir=OUT_DIR)
    try:
        procs = []
        objs = []
        for src in SOURCES:
            obj = os.path.join(tmp, src.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
            procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        log = []
        failed = []
        for src, cmd, p in procs:
            out, _ = p.communicate()
            text = out.decode(errors="replace")
            log.append("### %s\n%s\n%s" % (src, " ".join(cmd), text))
            if p.returncode != 0:
                failed.append(src)
        with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
            f.write("\n".join(log))
        if failed:
            sys.stderr.write("\n".join(log))
            raise RuntimeError("nvcc failed for %s" % ", ".join(failed))
        tmp_lib = os.path.join(tmp, "libmsm_g1.so")
        link = [nvcc, "-shared", "-o", tmp_lib] + objs + ARCH
        res = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + res.stdout.decode(errors="replace"))
        os.replace(tmp_lib, LIB)
        if verbose:
            print("\n".join(log))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
