/*
 * msm_g1_testing.h -- test hooks of libmsm_g1.so.  They run single device
 * primitives of the MSM path on arrays so that the tests can compare each
 * primitive with the CPU oracle.  Not needed to compute an MSM.
 *
 * All pointers are device pointers (16-byte aligned), arrays of n elements,
 * field elements as 8 x uint32 Montgomery limbs (< p), points as in msm_g1.h.
 * Calls are asynchronous on stream; they return 0 or a negative MSM_G1_ERR_*.
 */
#ifndef MSM_G1_TESTING_H
#define MSM_G1_TESTING_H

#include "msm_g1.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Field operations in F_p (the Montgomery multiplication the pages call the
 * "montgomery products", PR #23520, section "Why not split the inverse loop
 * too?"; the inversion is the one batched affine addition amortises, PR #23736,
 * section "Goal & lever"). */
#define MSM_G1_TEST_FQ_MUL 0 /* out = a * b           */
#define MSM_G1_TEST_FQ_SQR 1 /* out = a * a (the 36-product squaring of the batched additions) */
#define MSM_G1_TEST_FQ_ADD 2 /* out = a + b           */
#define MSM_G1_TEST_FQ_SUB 3 /* out = a - b           */
#define MSM_G1_TEST_FQ_NEG 4 /* out = -a              */
#define MSM_G1_TEST_FQ_INV 5 /* out = a^-1 (0 -> 0), safegcd divsteps (the MSM's inversion) */
#define MSM_G1_TEST_FQ_INV_FERMAT 6 /* out = a^(p-2) by square and multiply */
#define MSM_G1_TEST_FQ_INV_TABLE 7 /* out = a^-1 (0 -> 0), safegcd with four divsteps per table lookup (the
                                      accumulation kernels' per-thread inversion) */
#define MSM_G1_TEST_FQ_INV_BLOCK 8 /* out = a^-1 for nonzero a: the block-shared inversion of the
                                      accumulation kernels (128 values per block through one pass of 32
                                      inversions shared by two warps); a zero makes its block's results
                                      unspecified */
int msm_g1_test_fq(int op, const uint32_t *a, const uint32_t *b, uint32_t *out, size_t n, cudaStream_t stream);

/* Point operations.  JAC_* take and return Jacobian points (24 uint32),
 * MIXED adds a Jacobian a and an affine b, TO_AFFINE normalises a Jacobian a
 * into an affine out (16 uint32).  *_COOP are the cooperative doubling,
 * addition and mixed addition of the window combination (one warp per
 * element); *_COOP8 the same with one group of 8 lanes per element, as the
 * bucket reduction runs them (four elements per warp); DBL5_COOP one warp per
 * element. */
#define MSM_G1_TEST_JAC_DBL 0
#define MSM_G1_TEST_JAC_ADD 1
#define MSM_G1_TEST_JAC_MIXED 2
#define MSM_G1_TEST_TO_AFFINE 3
#define MSM_G1_TEST_JAC_DBL_COOP 4
#define MSM_G1_TEST_JAC_ADD_COOP 5
#define MSM_G1_TEST_JAC_MIXED_COOP 6
#define MSM_G1_TEST_JAC_DBL_COOP8 7
#define MSM_G1_TEST_JAC_ADD_COOP8 8
#define MSM_G1_TEST_JAC_MIXED_COOP8 9
#define MSM_G1_TEST_JAC_DBL5_COOP 10 /* five doublings in a row ([32] a) by the window combination's chain */
#define MSM_G1_TEST_AFF_ADD 11 /* a + b for affine a, b (16 words each) into Jacobian (the finish's first step) */
int msm_g1_test_g1(int op, const uint32_t *a, const uint32_t *b, uint32_t *out, size_t n, cudaStream_t stream);

/* The residue-number-system arithmetic of the window combination and the
 * bucket reduction's shifts (one block of two warps per element).  Field
 * values are positional Montgomery form (8 words), points positional Jacobian
 * (24 words), as in msm_g1_test_fq / msm_g1_test_g1.
 *   RNS_MUL       out = a * b, through the RNS (must equal MSM_G1_TEST_FQ_MUL)
 *   RNS_SQR_CHAIN out = a^(2^arg) by arg squarings in the RNS
 *   RNS_DBL_N     out = 2^arg a, by the two-warp projective doubling chain
 *   RNS_ADD       out = a + b by the complete projective addition (any a, b:
 *                 infinity, a = b and a = -b included)
 *   RNS_HORNER    a holds arg window sums per element (24 words each, window
 *                 0 first); out = sum_w 2^(13 w) T_w by Horner's rule
 *   RNS_IS_ZERO   a holds an integer below arg * p (8 words); out[i] = 1 if it
 *                 is a multiple of p, else 0 (one word per element) */
#define MSM_G1_TEST_RNS_MUL 0
#define MSM_G1_TEST_RNS_SQR_CHAIN 1
#define MSM_G1_TEST_RNS_DBL_N 2
#define MSM_G1_TEST_RNS_ADD 3
#define MSM_G1_TEST_RNS_HORNER 4
#define MSM_G1_TEST_RNS_IS_ZERO 5
int msm_g1_test_rns(int op, const uint32_t *a, const uint32_t *b, uint32_t *out, size_t n, int arg,
                    cudaStream_t stream);

/* Batched affine addition, the accumulation's inner step: out_i = a_i + b_i
 * for affine a, b (16 uint32 each), with one field inversion shared by each
 * run of batch_s consecutive pairs (batch_s as MSM_G1_PARAM_BATCH_S).
 * Equal, opposite and infinite operands are allowed.  mode bit 0 selects the
 * build the large accumulation launches use (the backward multiplications of
 * the batch inlined, 1) or the one of small launches (called, 0); bit 1 makes
 * the 128 threads of each block share one inversion as the accumulation
 * kernels do (2) instead of one inversion per thread (0).  Other mode values
 * are INVALID_ARG. */
int msm_g1_test_batch_add(const uint32_t *a, const uint32_t *b, uint32_t *out, size_t n, int batch_s,
                          int mode, cudaStream_t stream);

/* Signed window digits of n scalars (8 uint32 each) as the MSM forms them:
 * digits (n x W int32, W = ceil(nbits/c), window-major per scalar), nbits =
 * 255 for scalars reduced mod r (plain windows) or 128 for GLV halves (the
 * scalars must then be < 2^127).  With q = floor(nbits/W) and e = nbits - q W,
 * window w covers bits [off_w, off_w + c_w), c_w = q + 1 for the lowest e
 * windows and q for the others; each digit lies in (-2^(c_w - 1), 2^(c_w - 1)]
 * and sum_w digit_w 2^off_w = k (k mod r for nbits = 255). */
int msm_g1_test_digits(const uint32_t *scalars, size_t n, int c, int nbits, int32_t *digits, cudaStream_t stream);

/* GLV split of n scalars (8 uint32 each, reduced mod r first): out holds 10
 * uint32 per scalar, |k1| (4 limbs), |k2| (4 limbs), then the signs s1, s2
 * (1 = negative), with k = k1 + lambda k2 (mod r) and |k1|, |k2| < 2^127. */
int msm_g1_test_glv_split(const uint32_t *scalars, size_t n, uint32_t *out, cudaStream_t stream);

/* Host-only: the endomorphism constants the device code uses, beta in
 * Montgomery form (8 limbs; phi(x, y) = (beta x, y)) and lambda (8 limbs,
 * plain, phi = [lambda] on G1).  Touches no device. */
int msm_g1_glv_constants(uint32_t *beta_mont, uint32_t *lambda);

/* Copy an internal buffer of the last run to host memory (synchronises):
 * which = 0: bucket counts (W*B uint32), 1: even-padded bucket offsets
 * (W*B+1 uint32), 2: sorted entries (offset[W*B] uint32: point index with
 * bit 31 = negate, 0xffffffff = padding).  *bytes receives the buffer size;
 * at most max_bytes are copied. */
int msm_g1_debug_read(msm_g1_ctx *ctx, int which, void *host_dst, size_t max_bytes, size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* MSM_G1_TESTING_H */
