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

Inputs fit in L2 (129 MB), so L2 is flushed (a 256 MiB write) before every
timed step, outside the step's CUDA events.
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
# 64-bit multiply-add) takes two of those slots (measured on this GB300 by
# elliptic_curve_scalar_gb300/csrc/imad_rate.cu: mad.lo 18.7 Tops/s, paired
# lo/hi rows 8.9 T products/s).  A Montgomery multiplication on 8 x 32-bit
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


# The level-0 accumulation kernel's translation unit and every header it
# includes.  profiles/traffic.json holds ncu DRAM counters for one build of the
# kernel together with the digest of these files at that build; the bench line
# reports the counters as the roofline's traffic only while the digest matches.
LEVEL0_SOURCES = ("msm_accum.cu", "msm_internal.cuh", "msm_core.cuh", "g1_coop.cuh", "g1.cuh", "glv.cuh",
                  "inv.cuh", "fq.cuh")


def level0_sources_digest(read=None):
    """sha256 over LEVEL0_SOURCES (name and contents of each, in order);
    read(name) -> bytes supplies the contents (default: the working tree)."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "elliptic_curve_scalar_gb300", "csrc", name), "rb") as f:
                return f.read()
    h = hashlib.sha256()
    for name in LEVEL0_SOURCES:
        h.update(name.encode() + b"\0" + read(name) + b"\0")
    return h.hexdigest()


def level0_traffic(config_key, prof=None):
    """(traffic, earlier): the ncu DRAM bytes of the level-0 launch for this
    workload when they were taken on the kernel as it is now, else None and
    the figure of the earlier build (or None when there is none)."""
    prof = prof or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(prof) as f:
            tj = json.load(f)
    except (OSError, ValueError):
        return None, None
    val = tj.get(config_key)
    if val is None:
        return None, None
    if tj.get("sources_sha256") == level0_sources_digest():
        return val, None
    return None, val


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="n2p16", choices=sorted(CONFIGS))
    ap.add_argument("--c", type=int, default=0, help="override the window size")
    ap.add_argument("--batch-s", type=int, default=0,
                    help="additions per thread batch: 1..64, 0 = the library's choice (64)")
    ap.add_argument("--tpb", type=int, default=128)
    ap.add_argument("--finish", type=int, default=0, help="small-bucket threshold T (0 = automatic)")
    ap.add_argument("--groups", type=int, default=0, help="window groups of the pipelined schedule (0 = library default)")
    ap.add_argument("--glv", type=int, default=1, choices=[0, 1], help="split scalars by the GLV endomorphism")
    ap.add_argument("--inversion", type=int, default=0, choices=[0, 1], help="0: safegcd, 1: Fermat")
    ap.add_argument("--batch", type=int, default=1,
                    help="K > 1: each step is K independent MSMs of the workload's size, fused by msm_g1_run_batch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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

def oracle_points_per_s(cfg, sample, threads=None):
    """Time the CPU oracle (as it stands) on the first ``sample`` terms."""
    import oracle
    r, k = workload(dict(cfg, n=sample))
    pts = oracle.generator_multiples(r, threads=threads)
    threads = threads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.msm(pts, k, threads=threads)
    dt = time.perf_counter() - t0
    return sample / dt, dt, threads


def run_reference(args, cfg):
    world, rank, _ = dist_setup("gloo")
    if rank != 0:  # the oracle runs once, on rank 0; the other ranks leave without work
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    sample = 8192
    vals, times = [], []
    threads = None
    for i in range(args.warmup + args.steps):
        v, dt, threads = oracle_points_per_s(cfg, sample)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
    value = sample * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "points/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic",
        "config": {"workload": "BN254 G1 MSM %s, CPU oracle on the first %d terms per step" % (args.config, sample),
                   "n": cfg["n"], "c": cfg["c"], "kind": cfg["kind"], "seed": cfg["seed"]},
        "cpu_baseline": {"value": value, "unit": "points/s", "cores": threads, "kind": "oracle",
                         "sample": "first %d terms of the %s workload per step" % (sample, args.config)},
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


# ------------------------------------------------------------- GPU arm

def run_gpu(args, cfg):
    import torch
    from elliptic_curve_scalar_gb300 import msm as gm
    from elliptic_curve_scalar_gb300 import synth

    world, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = cfg["n"]
    c = args.c or cfg["c"]
    K = max(1, args.batch)
    r, k = workload(dict(cfg, n=K * n))  # K independent MSMs of n terms each (K = 1: the plain MSM)
    offsets = [i * n for i in range(K + 1)]

    ctx = gm.MsmG1(K * n, c, max_batch=K)
    ctx.set_param(gm.PARAM_BATCH_S, args.batch_s)
    ctx.set_param(gm.PARAM_TPB, args.tpb)
    ctx.set_param(gm.PARAM_FINISH, args.finish)
    ctx.set_param(gm.PARAM_GROUPS, args.groups)
    ctx.set_param(gm.PARAM_GLV, args.glv)
    ctx.set_param(gm.PARAM_INVERSION, args.inversion)
    scal_d = gm.to_device(synth.scalars_to_u32(k), dev)
    # points P_i = [r_i]G built on the device by the library's fixed-base kernel
    pts_d = ctx.mul_generator(gm.to_device(synth.scalars_to_u32(r), dev))
    out_d = torch.empty(24 * K, dtype=torch.int32, device=dev)

    def msm(p_in, s_in):  # one step: the MSM, or the K fused MSMs of a batch
        if K == 1:
            ctx.run(p_in, s_in, c, out=out_d)
        else:
            ctx.run_batch(p_in, s_in, offsets, c, out=out_d.view(K, 24))
    torch.cuda.synchronize()
    pts_h = pts_d.cpu().pin_memory()
    scal_h = scal_d.cpu().pin_memory()
    out_h = torch.empty(24, dtype=torch.int32).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # warm-up (also fixes the launch count and the exact work counters)
    ctx.set_param(gm.PARAM_STATS, 1)
    for _ in range(max(args.warmup, 3)):
        msm(pts_d, scal_d)
    stats = ctx.stats()
    nwin = -(-(gm.GLV_BITS if args.glv else gm.PLAIN_BITS) // c)
    counts, _ = ctx.debug_read(0, K * nwin * (1 << (c - 1)))
    ctx.set_param(gm.PARAM_STATS, 0)
    msm(pts_d, scal_d)
    launches_per_msm = int(ctx.stats()["launches"])

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    # timed region: K production MSMs (pipelined window groups), each bracketed
    # by CUDA events on the calling stream, which the library orders after all
    # of its internal streams
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(uuid)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.zero_()  # evict the inputs from L2 (outside the step's events)
        starts[s].record(stream)
        msm(pts_d, scal_d)
        ends[s].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = world * K * n * args.steps / (total_ms / 1000.0)

    # phase-timed steps: the serial schedule with CUDA events between phases on
    # the calling stream, which every kernel then runs on; the level-0 kernel's
    # duration for the roofline comes from these events
    ctx.set_param(gm.PARAM_TIMING, 1)
    phases = []
    for s in range(min(args.steps, 50)):
        flush.zero_()
        msm(pts_d, scal_d)
        phases.append(ctx.phase_ms())
    ctx.set_param(gm.PARAM_TIMING, 0)
    clocks = sampler.stop()

    # end to end through the C ABI with host buffers (msm_g1_run_host): every
    # step uploads that step's points and scalars from pinned host memory,
    # runs the MSM and downloads the 96-byte result
    ctx.set_param(gm.PARAM_TIMING, 0)
    e2e_steps = args.steps
    out_hk = torch.empty(24 * K, dtype=torch.int32).pin_memory()
    if K == 1:
        ctx.run_host(pts_h, scal_h, c, out=out_h)  # first call allocates the device copies
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        if K == 1:
            ctx.run_host(pts_h, scal_h, c, out=out_h)
        else:  # no host-buffer batch entry: torch uploads, msm_g1_run_batch, torch download
            msm(pts_h.to(dev, non_blocking=True), scal_h.to(dev, non_blocking=True))
            out_hk.copy_(out_d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    # roofline of the dominant kernel: level-0 batched affine accumulation
    m = counts.astype(np.int64)
    adds_l0 = int((m // 2).sum())            # pairs with two operands at level 0
    adds_total = int((m - (m > 0)).sum())    # every bucket of m entries needs m - 1 additions
    l0_ms = statistics.mean(p["accum_l0"] for p in phases)
    acc_ms = statistics.mean(p["accum_l0"] + p["accum_tree"] for p in phases)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    sm_max_mhz = peaks.get("sm_max_mhz", 2070.0)
    peak_timad = sms * IMAD_SLOTS_PER_CLK_PER_SM * sm_max_mhz * 1e6 / 1e12
    strict_imad = adds_l0 * IMAD_SLOTS_PER_ADD
    achieved = strict_imad / (l0_ms / 1e3) / 1e12
    traffic, traffic_earlier = level0_traffic("%s_S%s" % (args.config, args.batch_s or "auto"))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # a bounded sample: about 13 core-seconds of oracle work (0.8 s wall on 16 Grace cores)
        sample = 65536
        v, dt, threads = oracle_points_per_s(cfg, sample)
        cpu = {"value": v, "unit": "points/s", "cores": threads, "kind": "oracle",
               "sample": "first %d terms of the %s workload (%.1f s wall)" % (sample, args.config, dt)}

    if rank == 0:
        mean_phase = {kname: round(statistics.mean(p[kname] for p in phases), 4) for kname in phases[0]}
        line = {
            "metric": METRIC, "value": value, "unit": "points/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / (n / (PAGES_MS_LOGN16 / 1e3))) if n == (1 << 16) and K == 1 else None,
            "dtype": "u32", "data": "synthetic",
            "config": {"workload": "BN254 G1 MSM %sn=%d c=%d S=%s tpb=%d%s, %s points [r_i]G and scalars, seed %d"
                                   % ("%d fused x " % K if K > 1 else "", n, c, args.batch_s or "auto", args.tpb,
                                      " GLV" if args.glv else "", cfg["kind"], cfg["seed"]),
                       "n": n, "c": c, "S": args.batch_s or "auto", "tpb": args.tpb, "kind": cfg["kind"], "glv": args.glv,
                       "batch": K,
                       "finish_t": args.finish or "auto", "groups": args.groups,
                       "l2": "flushed before every timed step (256 MiB write)", "replicas": world},
            "ms_per_msm": ms_per_step / K,
            "ms_median": statistics.median(step_ms),
            "phase_ms": mean_phase,
            "serial_ms_per_msm": round(sum(mean_phase.values()), 4),
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_timad, "unit": "TIMADslot/s",
                         "frac": achieved / peak_timad, "traffic": traffic,
                         # counters of an earlier build of the kernel (its sources changed since
                         # the capture): context only, hence traffic is null
                         "traffic_earlier_build": traffic_earlier,
                         "kernel": "k_accum_level0",
                         "peak_basis": "%d SMs x %d IMAD slots/clk x %.0f MHz (sm_max_mhz of MEASURED_PEAKS.json)"
                                       % (sms, IMAD_SLOTS_PER_CLK_PER_SM, sm_max_mhz),
                         "count_basis": "5 Fq muls x 264 IMAD slots (128 full limb products at 2 slots + 8 low) + 1 squaring x 208 slots (36 + 64 full products + 8 low) per addition = 1528; inversion excluded",
                         "algorithmic_imad_slots_per_launch": strict_imad,
                         "adds_per_launch": adds_l0,
                         "inversion": "%s; each thread's batch of up to %s additions has one product to "
                                      "invert, and where threads hold two or more pairs the 128 threads of a "
                                      "block share one inversion pass (warp 0)" % (
                             "Fermat a^(p-2)" if args.inversion else "safegcd (Bernstein-Yang divsteps)",
                             args.batch_s or 64),
                         # the count the scope table names: 6 field multiplications of 136 full
                         # limb products (272 slots) per addition, inversions by divsteps adding
                         # no multiplications (Fermat runs report null here)
                         "frac_count_6x272": None if args.inversion else
                         adds_l0 * 6 * 272 / (l0_ms / 1e3) / 1e12 / peak_timad,
                         "accumulation_frac_all_levels": adds_total * IMAD_SLOTS_PER_ADD
                         / (acc_ms / 1e3) / 1e12 / peak_timad},
            "cpu_baseline": cpu,
            "e2e": {"value": world * K * n / (e2e_ms / 1e3), "unit": "points/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": int(pts_h.numel() * 4 + scal_h.numel() * 4),
                    "d2h_bytes_per_step": 96 * K},
            "gpu_launches": launches_per_msm * args.steps,
            "schedule": "timed steps: window groups pipelined over the library's streams; phase_ms and the roofline: serial phase-timed steps",
            "clocks": clocks,
            "work": {"entries": int(stats["entries"]), "adds": int(stats["adds"]),
                     "inversions": int(stats["inversions"]), "levels": int(stats["levels"]),
                     "max_bucket": int(stats["max_bucket"])},
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
