/*
 * msm_g1.h -- C ABI of libmsm_g1.so: BN254 G1 multi-scalar multiplication
 * Q = sum_i k_i * P_i on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the bucket-method MSM whose GPU kernels the source pages
 * tune: scalars are split into c-bit windows ("n=2^16, c=13", PR #23520
 * "cache dx + idx in ba_fused_super pref_scratch", section "Measurements"),
 * points are grouped by bucket (the sorted_bucket_list / sorted_count_list
 * buffers of PR #23738 "stream-walker S-sweep", section "What would actually
 * win"), bucket sums are built from batched affine additions that share one
 * field inversion per batch of S additions (PR #23736 "stream-walker --
 * amortize the field inversion via large S + private pref_scratch", section
 * "Goal & lever"), and the result must equal an independent CPU computation of
 * the same sum (PR #23736, section "Change (correct, landed)").  The curve is
 * BN254 G1: y^2 = x^3 + 3 over F_p, p = 0x30644e72...d87cfd47, generator
 * (1, 2), prime group order r = 0x30644e72...f0000001.
 *
 * Data layout (all device memory unless stated otherwise, little-endian
 * 32-bit limbs, 16-byte aligned base pointers):
 *   point, affine:   16 x uint32: x[8], y[8], each in Montgomery form
 *                    (x * 2^256 mod p), fully reduced (< p).  (0, 0) is the
 *                    point at infinity.  Inputs are not checked for being on
 *                    the curve; an off-curve input gives an unspecified point
 *                    (never a fault).
 *   scalar:          8 x uint32, a plain (not Montgomery) integer < 2^256.
 *                    Values >= r are allowed and act as k mod r, because every
 *                    point of E(F_p) has order dividing r.
 *   result, Jacobian: 24 x uint32: X[8], Y[8], Z[8] in Montgomery form,
 *                    representing (X/Z^2, Y/Z^3); Z = 0 is infinity.  The
 *                    point is exact; its Jacobian representative may differ
 *                    between runs (the order of a bucket's entries follows
 *                    the device's atomics), so compare results in affine form.
 *
 * Errors: every entry point returns 0 on success or a negative MSM_G1_ERR_*
 * code; argument errors are detected on the host before any device work is
 * queued.  Calls are asynchronous on the given stream unless stated otherwise;
 * a context is not thread-safe (one run at a time per context).  A call on a
 * context runs on the device the context was created on, whatever device is
 * current, and leaves the calling thread's current device as it found it; the
 * stream passed must belong to the context's device.
 */
#ifndef MSM_G1_H
#define MSM_G1_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSM_G1_OK 0
#define MSM_G1_ERR_INVALID_ARG (-1) /* null pointer, misaligned pointer, c out of range, bad key */
#define MSM_G1_ERR_CUDA (-2)        /* a CUDA call or kernel launch failed */
#define MSM_G1_ERR_CAPACITY (-3)    /* n or c needs more scratch than the context holds */
#define MSM_G1_ERR_ALLOC (-4)       /* device or host allocation failed at create */
#define MSM_G1_ERR_NO_DEVICE (-5)   /* no CUDA device, or not compute capability 10.3 */

#define MSM_G1_MAX_WINDOW 20

/* Tunable keys for msm_g1_set_param / msm_g1_get_param. */
#define MSM_G1_PARAM_BATCH_S 1 /* most additions a thread batches under one inversion: 1, 2, 4, 8, 16, 32, 64,
                                  or 0 = automatic (default, 64).  The pages' walkerS, additions per inversion
                                  (PR #23738 "stream-walker S-sweep", section "What landed here") */
#define MSM_G1_PARAM_TPB 2     /* threads per block of the accumulation kernels: 64, 128, 256, or 0 =
                                  automatic (default: 256 from 2^19 points, 128 below).  The pages' walkerTpb
                                  (same section) */
#define MSM_G1_PARAM_TIMING 3  /* 1: record CUDA events between phases (default 0) */
#define MSM_G1_PARAM_STATS 4   /* 1: count additions and inversions on the device (default 0) */
#define MSM_G1_PARAM_GROUPS 5  /* window groups pipelined over the context's streams: 1..4, 0 = automatic
                                  (default: 2, and 3 from 2^19 points); of two groups the top one takes
                                  floor((W + 2) / 4) of the W windows, otherwise they split evenly */
#define MSM_G1_PARAM_FINISH 6  /* buckets with at most T items leave the affine tree and are summed in
                                  Jacobian coordinates: T = 1..64, 1 = never, 0 = automatic (default) */
#define MSM_G1_PARAM_GLV 7     /* 1: split every scalar by the curve endomorphism (default), 0: plain windows */
#define MSM_G1_PARAM_INVERSION 8 /* field inversion of the batched additions: 0 = safegcd divsteps (default),
                                    1 = Fermat a^(p-2) (slower; kept for comparison) */
#define MSM_G1_PARAM_GRAPH 9   /* 1 (default): msm_g1_run of fewer than 2^19 points (and msm_g1_run_host, when
                                  its three host buffers are page-locked) captures its launches and copies as
                                  a CUDA graph on the context's own stream and replays it while the pointers,
                                  n, window_c and the parameters stay the same (setting any parameter drops
                                  the graph); 0: every run launches its kernels directly */
#define MSM_G1_PARAM_GRID 10   /* most blocks one accumulation launch may use (level 0 and every tree level):
                                  0 = automatic (default: whole resident waves for launches of fewer than four
                                  waves, else one block per tpb x S additions); a smaller cap makes each thread
                                  take several batches in turn.  The pages' walkerMaxWg, the cap on the
                                  walker's workgroups (PR #23736 "stream-walker -- amortize the field inversion
                                  via large S + private pref_scratch", section "Change (correct, landed)") */
#define MSM_G1_PARAM_ACC_PLACEMENT 11 /* where a batch keeps its S prefix products (the pages' pref_scratch,
                                  moved from workgroup to private memory in PR #23736, section "Change
                                  (correct, landed)"; PR #23738 "stream-walker S-sweep", section "What would
                                  actually win", asks to move it out again): MSM_G1_ACC_LOCAL (default),
                                  MSM_G1_ACC_SHARED or MSM_G1_ACC_REGISTERS (values below).  The placement
                                  bounds the batch size: shared 4..32 with S x 32 x TPB <= 200 KB, registers
                                  2..8; a request outside is clamped into that range */
#define MSM_G1_ACC_LOCAL 0     /* the thread's stack frame: device memory (HBM) cached in L1 and L2 */
#define MSM_G1_ACC_SHARED 1    /* the block's shared memory, S x 32 bytes per thread */
#define MSM_G1_ACC_REGISTERS 2 /* registers: the batch's loops unrolled so that every index is constant */

typedef struct msm_g1_ctx msm_g1_ctx;

/* Create a context on the current CUDA device and allocate its device
 * scratch (one allocation, owned by the context): the buffers the pages size
 * per configuration (PR #23738 "stream-walker S-sweep", section "What landed
 * here": "all S-dependent buffer sizing"), sized here once for the largest run.  Scratch covers every run
 * with n <= max_n and c <= max_c whose entry count (n * ceil(255/c) plain,
 * 2n * ceil(128/c) with the GLV split) is at most
 * max_n * max(ceil(255/c8), 2 ceil(128/c8)), c8 = min(8, max_c); every c >= c8
 * qualifies.  msm_g1_scratch_bytes gives the size.
 * max_c in [1, MSM_G1_MAX_WINDOW]; max_n in [1, 2^30].  Synchronous.
 * Returns MSM_G1_ERR_NO_DEVICE without a usable GPU, MSM_G1_ERR_ALLOC when the
 * allocation fails.  On error *ctx is set to NULL. */
int msm_g1_create(msm_g1_ctx **ctx, size_t max_n, int max_c);

/* No page counterpart (the pages run one MSM at a time).
 * As msm_g1_create, with the per-bucket and per-window buffers sized for
 * max_batch MSMs fused in one pass of msm_g1_run_batch (1 <= max_batch <=
 * 4096); max_n then bounds the terms of a whole pass.  msm_g1_create(ctx, n,
 * c) is msm_g1_create_batch(ctx, n, c, 1); a batch that does not fit one pass
 * runs as several. */
int msm_g1_create_batch(msm_g1_ctx **ctx, size_t max_n, int max_c, int max_batch);

/* The MSM the pages accelerate (see the file comment for its steps and sources).
 * Q = sum_{i<n} k_i * P_i, written to out_jacobian (device, 24 uint32).
 * With MSM_G1_PARAM_GLV = 1 (the default) each term is split by the
 * endomorphism phi(x, y) = (beta x, y) = [lambda](x, y) of BN254 G1 into
 * k1 P + k2 phi(P) with |k1|, |k2| < 2^127 (Gallant-Lambert-Vanstone), so the
 * bucket method runs over 2n terms with ceil(128/c) windows of c bits instead
 * of n terms with ceil(255/c) windows; the result is the same point.
 * The context's own streams run the window groups concurrently; they are
 * ordered after `stream` at the start and `stream` waits for them at the end,
 * so to the caller the call behaves like work queued on `stream`.
 * points_affine: device, n x 16 uint32 (layout above), read only.
 * scalars: device, n x 8 uint32, read only.
 * window_c: 1..max_c, or 0 to let the library choose (msm_g1_auto_window).
 * stream: the CUDA stream all work is queued on (0 = legacy default stream).
 * The caller owns inputs and output and must keep them alive until the stream
 * reaches the end of this call; the context's scratch is reused by the next
 * call.  n = 0 writes infinity.  No host synchronisation. */
int msm_g1_run(msm_g1_ctx *ctx, const uint32_t *points_affine, const uint32_t *scalars, size_t n,
               int window_c, uint32_t *out_jacobian, cudaStream_t stream);

/* No page counterpart: many MSMs fused into one pass.
 * A batch of count independent MSMs: out_jacobian[m] (24 uint32 each,
 * device) = sum over terms i in [offsets[m], offsets[m+1]) of k_i * P_i.
 * points_affine / scalars: device, the MSMs' terms concatenated (offsets[count]
 * terms, layouts as for msm_g1_run); offsets: HOST array of count + 1
 * nondecreasing term offsets with offsets[0] = 0 (empty MSMs give infinity).
 * The MSMs run fused -- one sort, one accumulation pass, one reduction over
 * the windows of all MSMs of a pass and one combination warp pair per MSM -- which
 * is what makes many small MSMs cheap; a batch larger than the context's
 * buffers is split into consecutive passes.  window_c applies to every MSM
 * (0: chosen for the largest one).  Each MSM must have at most max_n terms.
 * Asynchronous on stream; offsets may be reused as soon as the call returns. */
int msm_g1_run_batch(msm_g1_ctx *ctx, const uint32_t *points_affine, const uint32_t *scalars, const size_t *offsets,
                     int count, int window_c, uint32_t *out_jacobian, cudaStream_t stream);

/* The pages' "wall" time covers the whole call from the host (PR #23738,
 * section "Real-hardware data"); this entry point is that call.
 * The same MSM with inputs and output in HOST memory: points_affine (n x 16
 * uint32), scalars (n x 8 uint32) and out_jacobian (24 uint32), layouts as for
 * msm_g1_run.  The call queues, on `stream`, the upload of the scalars, the
 * MSM and the download of the result; the points are uploaded on one of the
 * context's own streams while the sort (which needs only the scalars) runs,
 * and the accumulation waits for them.  The first call allocates device
 * copies for max_n points and scalars (synchronous; MSM_G1_ERR_ALLOC on
 * failure).  With pinned (page-locked) host buffers every copy is
 * asynchronous and the caller reads out_jacobian after synchronising
 * `stream`; with pageable buffers CUDA stages the copies and may block.  The
 * host buffers must stay valid until the stream reaches the end of the call. */
int msm_g1_run_host(msm_g1_ctx *ctx, const uint32_t *points_affine, const uint32_t *scalars, size_t n,
                    int window_c, uint32_t *out_jacobian, cudaStream_t stream);

/* Workload builder: the pages' "independent points" (PR #23736, section
 * "Change (correct, landed)", which replaced an arithmetic progression of G).
 * out_i = [k_i]G for the generator G = (1, 2), as affine Montgomery points
 * (n x 16 uint32, infinity as (0, 0)).  scalars: device, n x 8 uint32, any
 * 256-bit value.  A utility for building workloads P_i = [r_i]G on the device;
 * it is not part of the MSM.  Asynchronous on stream. */
int msm_g1_mul_generator(msm_g1_ctx *ctx, const uint32_t *scalars, size_t n, uint32_t *out_points_affine,
                         cudaStream_t stream);

/* The same MSM as msm_g1_run, for callers that cannot allocate device memory
 * (their device heap is owned by another allocator, they run under a fixed
 * memory budget, or they cannot afford cudaMalloc's implicit synchronisation).
 * The source pages have no counterpart: this entry point exists for such
 * callers only.  No context: all scratch comes from one fixed 8 MiB array in
 * device global memory that the library holds on every GPU that loads it until
 * the process exits.  Limits: window_c <= 10.  With window_c in 8..10, or 0
 * (which picks a window within that range), any n <= 4096 fits.  A smaller
 * window needs more bucket entries per point (2 ceil(128 / c) with the GLV
 * split, against a fixed budget of 4096 x 32), so it fits proportionally fewer
 * points: n <= 3767 at c = 7, for instance.  Inputs beyond the limits return
 * MSM_G1_ERR_CAPACITY without device work.  The device-side capacity check
 * that msm_g1_last_stats reports for a context (out[7]) has no reader here;
 * the fixed sizing keeps it from ever firing.  The first call on a device looks up the array's device address on
 * that device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Every call reuses the same array: the calls clear what must start
 * at zero themselves, but calls whose device work overlaps (different streams,
 * or host threads, without ordering) race on the array and give wrong results.
 * Inputs, output and stream as for msm_g1_run; a GPU of compute capability
 * 10.3 is required (MSM_G1_ERR_NO_DEVICE otherwise). */
int msm_g1_run_noalloc(const uint32_t *points_affine, const uint32_t *scalars, size_t n, int window_c,
                       uint32_t *out_jacobian, cudaStream_t stream);

/* No page counterpart.  Release the context's scratch (synchronises the context's device first).
 * NULL is a no-op. */
void msm_g1_destroy(msm_g1_ctx *ctx);

/* The pages' MsmConfig runtime knobs (PR #23738, section "What landed here").
 * Set / read a tunable (MSM_G1_PARAM_*).  Takes effect on the next run. */
int msm_g1_set_param(msm_g1_ctx *ctx, int key, int value);
int msm_g1_get_param(const msm_g1_ctx *ctx, int key, int *value);

/* The pages' per-phase GPU times (the "stream_walker" phase beside the wall
 * time: PR #23736, section "Real-hardware results").
 * With MSM_G1_PARAM_TIMING = 1: wait for the last run and copy up to nphase
 * phase durations in milliseconds (decompose+histogram, scan, scatter,
 * accumulate level 0, accumulate levels >= 1, bucket reduction, window
 * combination) into ms.  Returns the number of phases written.  Timing runs
 * take the serial schedule (one stream, phases in order); otherwise the
 * phases of different window groups overlap on the context's own streams. */
int msm_g1_last_phase_ms(msm_g1_ctx *ctx, float *ms, int nphase);

/* The pages count inversions as total additions / S (PR #23736, section
 * "Change (correct, landed)"); these are the counters behind such figures.
 * Counters of the last run (waits for it): out[0] = bucket entries (non-zero
 * digits), out[1] = non-empty buckets, out[2] = largest bucket; with
 * MSM_G1_PARAM_STATS = 1 also out[3] = affine additions performed by the
 * accumulation, out[4] = field inversions it performed, out[5] = tree levels
 * that had work (zero otherwise); out[6] = kernels the last run launched;
 * out[7] = non-zero if a device-side capacity check failed (never expected);
 * the last run's plan: out[8] = small-bucket threshold T it used (1 = none),
 * out[9] = buckets per chunk of the bucket reduction, out[10] = window groups.
 * Returns the number of counters written (at most nout, at most 11). */
int msm_g1_last_stats(msm_g1_ctx *ctx, uint64_t *out, int nout);

/* Host-only helpers (no device work).  The window c is the pages' (c = 13 at
 * n = 2^16: PR #23520 "cache dx + idx in ba_fused_super pref_scratch", section
 * "Measurements"); the scratch size is their estimateMem (same page, section
 * "Summary"); strerror has no page counterpart. */
int msm_g1_window_count(int c);                      /* ceil(255 / c): signed windows for scalars reduced mod r
                                                        (without the GLV split; with it, ceil(128 / c)) */
int msm_g1_auto_window(size_t n);                    /* the window the library picks for window_c = 0 */
size_t msm_g1_scratch_bytes(size_t max_n, int max_c); /* device bytes msm_g1_create allocates */
const char *msm_g1_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MSM_G1_H */
