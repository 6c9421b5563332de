#!/usr/bin/env python3
"""Benchmark: BN254 G1 multi-scalar multiplication on GB300.

One step = one complete MSM (digits, sort, accumulation, bucket reduction,
window combination) over seeded synthetic inputs already resident in HBM.
Default workload: n = 2^16 points [r_i]G, uniform scalars, window c = 13
(the pages' "logn=16" shape; PR #23520 "cache dx + idx in ba_fused_super
pref_scratch", section "Measurements"; the pages' S = 8 is their phones'
optimum, here the library picks the batch size).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

A timed step runs R MSMs back to back (R chosen from the warm-up so that a
step lasts about 10 ms), each bracketed by its own CUDA events; L2 is flushed
(a 256 MiB write) before every MSM, outside its events, since the 2^16 inputs
fit in L2 (129 MB).  The output of the timed MSMs is checked against the closed
form [sum k_i r_i mod r]G (the points are P_i = [r_i]G), computed here with
Python integers.  The same measurement and check then run on the larger
configurations (n = 2^20, 2^22 and the adversarial 2^20 mix) into the line's
"per_config" block.

  python bench.py --profile K [--config NAME]   # K MSMs and nothing else (for ncu launch lists)
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per MSM and points/sec (BN254 G1, n=2^16..2^22); % of IMAD roofline"

CONFIGS = {
    "n2p10": dict(n=1 << 10, c=8, kind="uniform", seed=1001),
    "n2p16": dict(n=1 << 16, c=13, kind="uniform", seed=1002),
    "n2p20": dict(n=1 << 20, c=16, kind="uniform", seed=1003),
    "n2p22": dict(n=1 << 22, c=16, kind="uniform", seed=1004),
    "n2p20adv": dict(n=1 << 20, c=16, kind="adversarial", seed=1006),
    # larger than the pages' sizes (not bench defaults)
    "n2p23": dict(n=1 << 23, c=16, kind="uniform", seed=1007),
    "n2p24": dict(n=1 << 24, c=16, kind="uniform", seed=1008),
}

# Pages' own figure for this metric and workload: Apple M2 (WebGPU, Chrome 148),
# logn = 16, S = 8: 50.0 ms median MSM wall (PR #23738 "stream-walker S-sweep",
# section "Real-hardware data").  Context only, another machine.
PAGES_MS_LOGN16 = 50.0

# IMAD roofline.  Each SM issues 64 low-half 32-bit multiply-adds per clock
# (4 sub-partitions x 16 lanes); a full 32 x 32 -> 64-bit limb product (a
# lo/hi pair over the same operands in one carry chain, which issues as one
# 64-bit multiply-add) takes two of those slots (measured on this GB300 with a
# throughput probe: mad.lo 18.7 Tops/s, paired lo/hi rows 8.9 T products/s).  A Montgomery multiplication on 8 x 32-bit
# limbs needs 64 + 64 full products (a_i b_j, m_i p_j) and 8 low products
# m_i = t_i n': 2 * 128 + 8 = 264 slots, the fewest any schoolbook
# Montgomery multiplication can issue on this pipe.
IMAD_SLOTS_PER_CLK_PER_SM = 64
IMAD_SLOTS_PER_FQ_MUL = 2 * 128 + 8
# A squaring needs 28 off-diagonal + 8 diagonal full products and the 8 low
# products of the reduction: 2 * (36 + 64) + 8 = 208 slots.
IMAD_SLOTS_PER_FQ_SQR = 2 * (36 + 64) + 8
# 5M + 1S per batched affine addition (prefix, 2 backward, slope, x3 square, y3)
IMAD_SLOTS_PER_ADD = 5 * IMAD_SLOTS_PER_FQ_MUL + IMAD_SLOTS_PER_FQ_SQR
# Jacobian point operations of the bucket reduction and the window combination
# (Explicit-Formulas Database, a = 0): madd-2007-bl 7M + 4S, add-2007-bl
# 11M + 5S, dbl-2009-l 2M + 5S; squarings counted at the dedicated squaring's
# slots (the strict count: the library's Jacobian chains square by multiplying)
IMAD_SLOTS_MADD = 7 * IMAD_SLOTS_PER_FQ_MUL + 4 * IMAD_SLOTS_PER_FQ_SQR
IMAD_SLOTS_JADD = 11 * IMAD_SLOTS_PER_FQ_MUL + 5 * IMAD_SLOTS_PER_FQ_SQR
IMAD_SLOTS_JDBL = 2 * IMAD_SLOTS_PER_FQ_MUL + 5 * IMAD_SLOTS_PER_FQ_SQR

# the phases of msm_g1_last_phase_ms whose work is field arithmetic, and their kernels
IMAD_PHASES = {
    "accum_l0": "k_accum_level0 (+ _wide)",
    "accum_tree": "k_accum_list (+ _wide), one launch per tree level",
    "bucket_reduce": "k_finish_chunks (or k_finish + k_reduce_chunks), k_reduce_jobs, k_reduce_shift, k_reduce_final",
    "combine": "k_combine_part",
}
# the larger configurations measured into the line's per_config block
PER_CONFIG = ("n2p20", "n2p22", "n2p20adv")
# BN254 (G1 over F_p, scalars mod r) for the closed-form check of the timed output
FQ_P = 0x30644e72e131a029b85045b68181585d97816a916871ca8d3c208c16d87cfd47
FR_R = 0x30644e72e131a029b85045b68181585d2833e84879b9709143e1f593f0000001


# The library's kernel sources.  profiles/traffic.json holds ncu DRAM counters
# (bytes per MSM, per phase, per workload) for one build together with the
# digest of these files' code at that build; the bench line reports the
# counters only while the digest matches (any code change makes them stale,
# an edited comment does not).
KERNEL_SOURCES = ("msm_g1.cu", "msm_accum.cu", "msm_internal.cuh", "msm_core.cuh", "g1_coop.cuh", "g1_proj.cuh",
                  "rns.cuh", "rns_consts.cuh", "g1.cuh", "glv.cuh", "inv.cuh", "divstep_table.cuh", "fq.cuh")


def code_only(src):
    """C/C++ source bytes without comments, whitespace runs collapsed to one
    space (string and character literals kept as they are): what the compiler
    sees, so that an edited comment leaves the digest below unchanged."""
    out, i, n = bytearray(), 0, len(src)

    def space():
        if out and out[-1] != 0x20:
            out.append(0x20)

    while i < n:
        c = src[i:i + 1]
        if src.startswith(b"//", i):
            j = src.find(b"\n", i)
            i = n if j < 0 else j
        elif src.startswith(b"/*", i):
            j = src.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
            space()
        elif c in (b'"', b"'"):
            j = i + 1
            while j < n and src[j:j + 1] != c:
                j += 2 if src[j:j + 1] == b"\\" else 1
            out += src[i:j + 1]
            i = j + 1
        elif c.isspace():
            j = i
            while j < n and src[j:j + 1].isspace():
                j += 1
            space()
            i = j
        else:
            out += c
            i += 1
    return bytes(out).strip()


def kernel_sources_digest(read=None):
    """sha256 over KERNEL_SOURCES (name and code of each, in order, comments
    left out: code_only); read(name) -> bytes supplies the contents (default:
    the working tree)."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "elliptic_curve_scalar_gb300", "csrc", name), "rb") as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode() + b"\0" + code_only(read(name)) + b"\0")
    return h.hexdigest()


def phase_traffic(config_key, phase, prof=None):
    """(bytes, stale): the ncu DRAM bytes per MSM of the phase's kernels for
    this workload when they were taken on the kernels as they are now (else
    None), and the stored figure when it belongs to another build (else None)."""
    prof = prof or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(prof) as f:
            tj = json.load(f)
    except (OSError, ValueError):
        return None, None
    val = tj.get("bytes_per_msm", {}).get(config_key, {}).get(phase)
    if val is None:
        return None, None
    if tj.get("sources_sha256") == kernel_sources_digest():
        return val, None
    return None, val


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="n2p16", choices=sorted(CONFIGS))
    ap.add_argument("--c", type=int, default=0, help="override the window size")
    ap.add_argument("--batch-s", type=int, default=0,
                    help="additions per thread batch: 1..64, 0 = the library's choice (64)")
    ap.add_argument("--tpb", type=int, default=0, help="threads per accumulation block (0 = the library's choice)")
    ap.add_argument("--place", type=int, default=0, choices=[0, 1, 2],
                    help="prefix products of a batch: 0 thread-local (device memory), 1 shared memory, 2 registers")
    ap.add_argument("--grid", type=int, default=0, help="most blocks per accumulation launch (0 = automatic)")
    ap.add_argument("--finish", type=int, default=0, help="small-bucket threshold T (0 = automatic)")
    ap.add_argument("--groups", type=int, default=0, help="window groups of the pipelined schedule (0 = library default)")
    ap.add_argument("--glv", type=int, default=1, choices=[0, 1], help="split scalars by the GLV endomorphism")
    ap.add_argument("--inversion", type=int, default=0, choices=[0, 1], help="0: safegcd, 1: Fermat")
    ap.add_argument("--batch", type=int, default=1,
                    help="K > 1: each step is K independent MSMs of the workload's size, fused by msm_g1_run_batch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per_config block")
    ap.add_argument("--reps", type=int, default=0, help="MSMs per timed step (0: about 10 ms per step)")
    ap.add_argument("--profile", type=int, default=0,
                    help="K > 0: run K MSMs of the configuration and exit (for ncu launch lists)")
    return ap.parse_args()


def dist_setup(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x, world, device=None):
    """The largest of the ranks' values of x: every replica's time counts, so the
    job is as slow as its slowest rank (x itself when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload(cfg):
    from elliptic_curve_scalar_gb300 import synth
    return synth.workload(cfg["kind"], cfg["n"], cfg["seed"])


# ------------------------------------------------------------ CPU oracle

def oracle_points_per_s(cfg, sample, threads=None, min_seconds=0.0):
    """Time the CPU oracle (as it stands) on the workload's first ``sample``
    points, the whole MSM repeated until ``min_seconds`` have passed; returns
    (points/s, seconds, threads, repetitions)."""
    import oracle
    r, k = workload(dict(cfg, n=sample))
    pts = oracle.generator_multiples(r, threads=threads)
    threads = threads or oracle.default_threads()
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.msm(pts, k, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return sample * reps / dt, dt, threads, reps


def run_reference(args, cfg):
    world, rank, _ = dist_setup("gloo")
    if rank != 0:  # the oracle runs once, on rank 0; the other ranks leave without work
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    sample = min(8192, cfg["n"])
    vals, times = [], []
    threads = None
    for i in range(args.warmup + args.steps):
        v, dt, threads, _ = oracle_points_per_s(cfg, sample)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
    value = sample * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "points/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic",
        "config": {"workload": "BN254 G1 MSM %s, CPU oracle on the first %d points per step" % (args.config, sample),
                   "n": cfg["n"], "c": cfg["c"], "kind": cfg["kind"], "seed": cfg["seed"]},
        "cpu_baseline": {"value": value, "unit": "points/s", "cores": threads, "kind": "oracle",
                         "sample": "first %d points of the %s workload per step" % (sample, args.config)},
        "e2e": {"value": value, "unit": "points/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None, tmpdir=None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False, dir=tmpdir)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.close()
        with open(self.file.name) as f:
            lines = f.readlines()
        os.unlink(self.file.name)
        return summarize_clocks(lines)


def summarize_clocks(lines):
    """The bench line's "clocks" from nvidia-smi rows of ClockSampler.FIELDS
    (csv, no header, no units): median SM clock, highest maximum clock, and
    every throttle reason seen active in any sample."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) == 9:
            rows.append(parts)
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].lower().startswith("active")})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------- closed-form check (host)

def dot_mod_r(k, r, chunk=1 << 18):
    """sum_i k_i r_i mod r for uint64[n, 4] scalar arrays.  8-bit limbs: each
    limb product is below 2^16 and a column sum over a chunk of 2^18 terms below
    2^34, exact in float64, so a BLAS matrix product gives every column sum."""
    kb = np.ascontiguousarray(k).view(np.uint8).reshape(k.shape[0], -1)
    rb = np.ascontiguousarray(r).view(np.uint8).reshape(r.shape[0], -1)
    cols = np.zeros((kb.shape[1], rb.shape[1]), dtype=np.int64)
    for i in range(0, kb.shape[0], chunk):
        cols += (kb[i:i + chunk].astype(np.float64).T @ rb[i:i + chunk].astype(np.float64)).astype(np.int64)
    s = 0
    for a in range(cols.shape[0]):
        for b in range(cols.shape[1]):
            s += int(cols[a, b]) << (8 * (a + b))
    return s % FR_R


def _aff_add(a, b):
    """chord-and-tangent law on y^2 = x^3 + 3 over F_p (None = infinity)"""
    if a is None:
        return b
    if b is None:
        return a
    if a[0] == b[0]:
        if (a[1] + b[1]) % FQ_P == 0:
            return None
        lam = 3 * a[0] * a[0] * pow(2 * a[1], FQ_P - 2, FQ_P) % FQ_P
    else:
        lam = (b[1] - a[1]) * pow(b[0] - a[0], FQ_P - 2, FQ_P) % FQ_P
    x = (lam * lam - a[0] - b[0]) % FQ_P
    return x, (lam * (a[0] - x) - a[1]) % FQ_P


def generator_multiple(s):
    """[s]G for G = (1, 2), affine, by double-and-add"""
    acc, base = None, (1, 2)
    while s:
        if s & 1:
            acc = _aff_add(acc, base)
        base = _aff_add(base, base)
        s >>= 1
    return acc


def jacobian_words_to_affine(words):
    """24 uint32 words (X, Y, Z, Montgomery form) -> affine (x, y) or None"""
    w = [int(v) for v in np.asarray(words, dtype=np.uint32).reshape(24)]
    X, Y, Z = (sum(w[8 * j + i] << (32 * i) for i in range(8)) for j in range(3))
    rinv = pow(1 << 256, FQ_P - 2, FQ_P)
    X, Y, Z = X * rinv % FQ_P, Y * rinv % FQ_P, Z * rinv % FQ_P
    if Z == 0:
        return None
    zi = pow(Z, FQ_P - 2, FQ_P)
    return X * zi * zi % FQ_P, Y * zi * zi * zi % FQ_P


def closed_form_ok(out_words, r, k, K, n):
    """Every result of the K MSMs of n terms equals [sum k_i r_i mod r]G."""
    outs = np.asarray(out_words, dtype=np.uint32).reshape(K, 24)
    for m in range(K):
        s = dot_mod_r(k[m * n:(m + 1) * n], r[m * n:(m + 1) * n])
        if jacobian_words_to_affine(outs[m]) != generator_multiple(s):
            return False
    return True


# ------------------------------------------------------ work per phase

def phase_work(counts, stats, c, glv, K):
    """IMAD issue slots of the strict algorithmic count of each field-arithmetic
    phase of one pass (K fused MSMs), from the bucket sizes and the plan the
    library reports for the run (small-bucket threshold T, chunk length L)."""
    nbits = 128 if glv else 255
    W = -(-nbits // c)
    q = nbits // W
    B = 1 << (c - 1)
    m = counts.astype(np.int64).reshape(K * W, B)
    adds_l0 = int((m // 2).sum())
    adds_tree = max(0, int(stats["adds"]) - adds_l0)
    # small-bucket finish: a bucket of h level-1 items leaves the tree with
    # ceil(h / stride) <= T items, summed by mixed additions
    T = int(stats.get("finish_t", 1)) or 1
    h = (m + 1) // 2
    items = h.copy()
    stride = np.ones_like(h)
    while True:
        big = items > T
        if not big.any():
            break
        stride = np.where(big, stride * 2, stride)
        items = np.where(big, -(-h // stride), items)
    jac = (items >= 2) & (T >= 2)
    madd = int(np.where(jac, items - 1, 0).sum())
    # chunk running sums: run += bucket (mixed, or full for a Jacobian bucket sum), sum += run,
    # both from the chunk's top bucket down; the first non-trivial addition of each starts from infinity
    L = int(stats.get("chunk_len", 4)) or 4
    G = B // L
    ne = (m > 0).reshape(K * W, G, L)[:, :, ::-1]
    jc = jac.reshape(K * W, G, L)[:, :, ::-1]
    has = ne.any(axis=2)
    first = np.where(has, ne.argmax(axis=2), L)
    first_jac = np.take_along_axis(jc, np.minimum(first, L - 1)[:, :, None], axis=2)[:, :, 0] & has
    madd += int((ne & ~jc).sum()) - int((has & ~first_jac).sum())
    jadd = int((ne & jc).sum()) - int(first_jac.sum()) + int(np.maximum(L - first - 1, 0).sum())
    # per window: job 0 sums the G chunk sums, job 1 + t the G/2 running sums with bit t set,
    # each job's value is doubled to its weight, then a tree over the jobs
    lg = G.bit_length() - 1
    Lg = L.bit_length() - 1
    jadd += K * W * ((G - 1) + lg * (G // 2 - 1) + lg)
    jdbl = K * W * sum(t - 1 + Lg for t in range(1, lg + 1))
    # Horner's rule over the windows: one doubling per bit below the top window, one addition per window
    cdbl = K * (nbits - q)
    cadd = K * (W - 1)
    return {
        "adds_l0": adds_l0, "adds_tree": adds_tree,
        "slots": {
            "accum_l0": adds_l0 * IMAD_SLOTS_PER_ADD,
            "accum_tree": adds_tree * IMAD_SLOTS_PER_ADD,
            "bucket_reduce": madd * IMAD_SLOTS_MADD + jadd * IMAD_SLOTS_JADD + jdbl * IMAD_SLOTS_JDBL,
            "combine": cdbl * IMAD_SLOTS_JDBL + cadd * IMAD_SLOTS_JADD,
        },
        "point_ops": {"bucket_reduce": {"madd": madd, "add": jadd, "dbl": jdbl},
                      "combine": {"dbl": cdbl, "add": cadd}},
    }


# ------------------------------------------------------------- GPU arm

def imad_peak(dev):
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return sms * IMAD_SLOTS_PER_CLK_PER_SM * mhz * 1e6 / 1e12, \
        "%d SMs x %d IMAD slots/clk x %.0f MHz (sm_max_mhz of MEASURED_PEAKS.json)" % (
            sms, IMAD_SLOTS_PER_CLK_PER_SM, mhz)


def make_context(args, cfg, dev, K, n):
    import torch
    from elliptic_curve_scalar_gb300 import msm as gm
    from elliptic_curve_scalar_gb300 import synth
    c = args.c or cfg["c"]
    r, k = workload(dict(cfg, n=K * n))  # K independent MSMs of n terms each (K = 1: the plain MSM)
    ctx = gm.MsmG1(K * n, c, max_batch=K)
    ctx.set_param(gm.PARAM_BATCH_S, args.batch_s)
    ctx.set_param(gm.PARAM_TPB, args.tpb)
    ctx.set_param(gm.PARAM_FINISH, args.finish)
    ctx.set_param(gm.PARAM_GROUPS, args.groups)
    ctx.set_param(gm.PARAM_GLV, args.glv)
    ctx.set_param(gm.PARAM_INVERSION, args.inversion)
    ctx.set_param(gm.PARAM_ACC_PLACEMENT, args.place)
    ctx.set_param(gm.PARAM_GRID, args.grid)
    scal_d = gm.to_device(synth.scalars_to_u32(k), dev)
    # points P_i = [r_i]G built on the device by the library's fixed-base kernel
    pts_d = ctx.mul_generator(gm.to_device(synth.scalars_to_u32(r), dev))
    out_d = torch.empty(24 * K, dtype=torch.int32, device=dev)
    offsets = [i * n for i in range(K + 1)]

    def msm(p_in, s_in):  # one MSM, or the K fused MSMs of a batch
        if K == 1:
            ctx.run(p_in, s_in, c, out=out_d)
        else:
            ctx.run_batch(p_in, s_in, offsets, c, out=out_d.view(K, 24))
    return ctx, c, r, k, pts_d, scal_d, out_d, msm


def measure(args, cfg, dev, world, K, n, with_e2e, sampler_uuid=None):
    """Warm-up, the timed steps, the phase-timed steps and the closed-form check
    of one configuration; returns (record, ctx, extras)."""
    import torch
    from elliptic_curve_scalar_gb300 import msm as gm

    ctx, c, r, k, pts_d, scal_d, out_d, msm = make_context(args, cfg, dev, K, n)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # warm-up (also fixes the launch count, the exact work counters and the plan)
    ctx.set_param(gm.PARAM_STATS, 1)
    for _ in range(max(args.warmup, 3)):
        msm(pts_d, scal_d)
    stats = ctx.stats()
    nwin = -(-(gm.GLV_BITS if args.glv else gm.PLAIN_BITS) // c)
    counts, _ = ctx.debug_read(0, K * nwin * (1 << (c - 1)))
    ctx.set_param(gm.PARAM_STATS, 0)
    torch.cuda.synchronize()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    msm(pts_d, scal_d)
    w1.record(stream)
    torch.cuda.synchronize()
    launches_per_msm = int(ctx.stats()["launches"])
    reps = args.reps or max(1, min(64, int(10.0 / max(w0.elapsed_time(w1), 1e-3))))

    # timed region: steps x reps production MSMs (pipelined window groups),
    # each bracketed by CUDA events on the calling stream, which the library
    # orders after all of its internal streams; L2 flushed before each
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(sampler_uuid) if sampler_uuid is not False else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        msm(pts_d, scal_d)
        b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    msm_ms = [a.elapsed_time(b) for a, b in ev]
    parity = closed_form_ok(gm.to_host(out_d), r, k, K, n)
    total_ms = max_over_ranks(sum(msm_ms), world, dev)

    # phase-timed MSMs: the serial schedule with CUDA events between phases on
    # the calling stream, which every kernel then runs on
    ctx.set_param(gm.PARAM_TIMING, 1)
    phases = []
    for _ in range(min(args.steps * reps, 50)):
        flush.zero_()
        msm(pts_d, scal_d)
        phases.append(ctx.phase_ms())
    ctx.set_param(gm.PARAM_TIMING, 0)
    clocks = sampler.stop() if sampler else None

    peak, peak_basis = imad_peak(dev)
    work = phase_work(counts, stats, c, args.glv, K)
    mean_phase = {kname: statistics.mean(p[kname] for p in phases) for kname in phases[0]}
    frac = {ph: work["slots"][ph] / (mean_phase[ph] / 1e3) / 1e12 / peak for ph in IMAD_PHASES}
    acc_ms = mean_phase["accum_l0"] + mean_phase["accum_tree"]
    rec = {
        "ms_per_msm": total_ms / (args.steps * reps * K),
        "ms_median": statistics.median(msm_ms) / K,
        "points_per_s": world * K * n * args.steps * reps / (total_ms / 1e3),
        "reps_per_step": reps,
        "parity": bool(parity),
        "phase_ms": {kname: round(v, 4) for kname, v in mean_phase.items()},
        "serial_ms_per_msm": round(sum(mean_phase.values()) / K, 4),
        "imad_frac": {ph: round(v, 4) for ph, v in frac.items()},
        "level0_frac": frac["accum_l0"],
        # every affine addition the accumulation kernels performed (device count), over level 0 and the tree
        "accumulation_frac_all_levels": int(stats["adds"]) * IMAD_SLOTS_PER_ADD / (acc_ms / 1e3) / 1e12 / peak,
        "work": {"entries": int(stats["entries"]), "adds": int(stats["adds"]), "adds_l0": work["adds_l0"],
                 "inversions": int(stats["inversions"]), "levels": int(stats["levels"]),
                 "max_bucket": int(stats["max_bucket"]), "finish_t": int(stats.get("finish_t", 0)),
                 "chunk_len": int(stats.get("chunk_len", 0)), "groups": int(stats.get("groups", 0)),
                 "point_ops": work["point_ops"]},
    }
    extras = dict(ctx=ctx, c=c, msm=msm, pts_d=pts_d, scal_d=scal_d, out_d=out_d, stream=stream, work=work,
                  mean_phase=mean_phase, frac=frac, peak=peak, peak_basis=peak_basis, clocks=clocks,
                  launches_per_msm=launches_per_msm, steps_msms=args.steps * reps, total_ms=total_ms)
    return rec, extras


def run_profile(args, cfg):
    """K MSMs of the configuration and nothing else, for ncu launch lists:
    per-kernel totals divided by K give the kernels' work per MSM.  The
    workload set-up launches k_gen_table_jac, k_gen_table_norm and
    k_mul_generator once before them."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    ctx, c, r, k, pts_d, scal_d, out_d, msm = make_context(args, cfg, dev, 1, cfg["n"])
    for _ in range(args.profile):
        msm(pts_d, scal_d)
    torch.cuda.synchronize()
    from elliptic_curve_scalar_gb300 import msm as gm
    ok = closed_form_ok(gm.to_host(out_d), r, k, 1, cfg["n"])
    print(json.dumps({"profile_msms": args.profile, "config": args.config, "parity": ok}), flush=True)
    ctx.close()
    return 0 if ok else 1


def run_gpu(args, cfg):
    import torch
    from elliptic_curve_scalar_gb300 import msm as gm

    world, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = cfg["n"]
    K = max(1, args.batch)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    rec, x = measure(args, cfg, dev, world, K, n, True, uuid)
    ctx, c, msm, stream = x["ctx"], x["c"], x["msm"], x["stream"]

    # end to end through the C ABI with host buffers (msm_g1_run_host): every
    # step uploads that step's points and scalars from pinned host memory,
    # runs the MSM and downloads the 96-byte result
    pts_h = x["pts_d"].cpu().pin_memory()
    scal_h = x["scal_d"].cpu().pin_memory()
    out_h = torch.empty(24, dtype=torch.int32).pin_memory()
    out_hk = torch.empty(24 * K, dtype=torch.int32).pin_memory()
    e2e_msms = x["steps_msms"]
    if K == 1:
        ctx.run_host(pts_h, scal_h, c, out=out_h)  # first call allocates the device copies
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_msms):
        if K == 1:
            ctx.run_host(pts_h, scal_h, c, out=out_h)
        else:  # no host-buffer batch entry: torch uploads, msm_g1_run_batch, torch download
            msm(pts_h.to(dev, non_blocking=True), scal_h.to(dev, non_blocking=True))
            out_hk.copy_(x["out_d"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_msms, world, dev)
    ctx.close()
    del x["pts_d"], x["scal_d"], x["out_d"]
    torch.cuda.empty_cache()

    # the roofline of the dominant field-arithmetic phase (largest serial time)
    mp, frac, peak = x["mean_phase"], x["frac"], x["peak"]
    dom = max(IMAD_PHASES, key=lambda ph: mp[ph])
    traffic, traffic_stale = phase_traffic(args.config, dom)
    achieved = frac[dom] * peak
    roofline = {
        "bound": "alu", "achieved": achieved, "peak": peak, "unit": "TIMADslot/s", "frac": frac[dom],
        "traffic": traffic, "traffic_other_build": traffic_stale,
        "phase": dom, "kernel": IMAD_PHASES[dom],
        "peak_basis": x["peak_basis"],
        "count_basis": "strict algorithmic IMAD issue slots: an Fq multiplication 264 (128 full limb products "
                       "at 2 slots + 8 low), a squaring 208; batched affine addition 5M + 1S = 1528, "
                       "madd-2007-bl 7M + 4S, add-2007-bl 11M + 5S, dbl-2009-l 2M + 5S; inversions excluded",
        "algorithmic_imad_slots_per_msm": x["work"]["slots"][dom] / K,
        "phase_ms_per_msm": mp[dom] / K,
        "frac_by_phase": rec["imad_frac"],
        "level0": {
            "frac": rec["level0_frac"],
            "adds_per_launch": rec["work"]["adds_l0"],
            # the scope table's count: 6 field multiplications of 136 full limb
            # products (272 slots) per addition; divsteps add none
            "frac_count_6x272": None if args.inversion else
            rec["work"]["adds_l0"] * 6 * 272 / (mp["accum_l0"] / 1e3) / 1e12 / peak,
            "inversion": "%s; each thread's batch of up to %s additions has one product to invert, and where "
                         "threads hold two or more pairs the 128 threads of a block share one inversion pass" % (
                             "Fermat a^(p-2)" if args.inversion else "safegcd (Bernstein-Yang divsteps)",
                             args.batch_s or 64),
        },
        "accumulation_frac_all_levels": rec["accumulation_frac_all_levels"],
    }

    per_config = None
    if K == 1 and not args.no_per_config:
        per_config = {}
        pc_sampler = ClockSampler(uuid) if rank == 0 else None
        for name in PER_CONFIG:
            if name == args.config:
                continue
            pc = CONFIGS[name]
            r2, x2 = measure(args, pc, dev, world, 1, pc["n"], False, False)
            x2["ctx"].close()
            lt, lt_stale = phase_traffic(name, "accum_l0")
            r2.update({"n": pc["n"], "c": args.c or pc["c"], "kind": pc["kind"], "seed": pc["seed"],
                       "level0_traffic": lt, "level0_traffic_other_build": lt_stale})
            per_config[name] = r2
            del x2
            torch.cuda.empty_cache()
        if pc_sampler:
            # the larger configurations run back to back on a GPU already warm from
            # the headline: their own clock record (a 2^20 MSM measured first in a
            # fresh process runs 3.39 ms, measured here after the headline 3.60 ms)
            per_config["clocks"] = pc_sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # a bounded sample: at most 2^16 of the workload's points (about 13
        # core-seconds of oracle work, 0.8 s wall on 16 Grace cores), smaller
        # workloads whole and repeated for half a second at least
        sample = min(65536, cfg["n"])
        v, dt, threads, reps = oracle_points_per_s(cfg, sample, min_seconds=0.5)
        cpu = {"value": v, "unit": "points/s", "cores": threads, "kind": "oracle",
               "sample": "first %d points of the %s workload, %d MSM(s) (%.1f s wall)" % (sample, args.config,
                                                                                    reps, dt)}

    if rank == 0:
        steps_msms = x["steps_msms"]
        reps = rec["reps_per_step"]
        ms_per_step = x["total_ms"] / args.steps
        line = {
            "metric": METRIC, "value": rec["points_per_s"], "unit": "points/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": (rec["points_per_s"] / (n / (PAGES_MS_LOGN16 / 1e3))) if n == (1 << 16) and K == 1
            else None,
            "dtype": "u32", "data": "synthetic",
            "config": {"workload": "BN254 G1 MSM %sn=%d c=%d S=%s tpb=%s%s, %s points [r_i]G and scalars, seed %d"
                                   % ("%d fused x " % K if K > 1 else "", n, c, args.batch_s or "auto", args.tpb or "auto",
                                      " GLV" if args.glv else "", cfg["kind"], cfg["seed"]),
                       "n": n, "c": c, "S": args.batch_s or "auto", "tpb": args.tpb or "auto", "kind": cfg["kind"],
                       "glv": args.glv, "batch": K, "finish_t": args.finish or "auto", "groups": args.groups,
                       "placement": ("local", "shared", "registers")[args.place], "grid": args.grid or "auto",
                       "msms_per_step": reps * K,
                       "l2": "flushed before every timed MSM (256 MiB write, outside its events)",
                       "replicas": world},
            "ms_per_msm": rec["ms_per_msm"],
            "ms_median": rec["ms_median"],
            "parity": rec["parity"],
            "phase_ms": rec["phase_ms"],
            "serial_ms_per_msm": rec["serial_ms_per_msm"],
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": world * K * n / (e2e_ms / 1e3), "unit": "points/s", "ms_per_msm": e2e_ms,
                    "h2d_bytes_per_step": int(pts_h.numel() * 4 + scal_h.numel() * 4) * reps,
                    "d2h_bytes_per_step": 96 * K * reps},
            "gpu_launches": x["launches_per_msm"] * steps_msms,
            "schedule": "timed MSMs: window groups pipelined over the library's streams; phase_ms and the "
                        "roofline: serial phase-timed MSMs",
            "clocks": x["clocks"],
            "work": rec["work"],
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.profile:
        return run_profile(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
