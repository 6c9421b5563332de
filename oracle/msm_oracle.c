/*
 * msm_oracle.c -- plain, slow, CPU reference for the BN254 G1 multi-scalar
 * multiplication Q = sum_i k_i * P_i.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load, link or
 * call this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or constant table with
 * the CUDA library: it uses its own radix (4 x 64-bit limbs), keeps residues
 * canonical (never Montgomery form except when asked to encode/decode), reduces
 * by Barrett's method (Handbook of Applied Cryptography, Algorithm 14.42) and
 * uses textbook Jacobian formulas, none of which the GPU path uses.
 *
 * What it computes follows the definition the pages rely on: the MSM result is
 * the group sum of the individual scalar multiples (PR #23736 "stream-walker --
 * amortize the field inversion via large S + private pref_scratch", section
 * "Change (correct, landed)": the GPU output is accepted when it equals an
 * independent CPU library's MSM).  The curve is BN254 G1 (y^2 = x^3 + 3 over
 * F_p), fixed by the workload definition because the pages never name it.
 *
 * Point format at this interface: 8 uint64 per point, x[4] then y[4], little
 * endian limbs, canonical residues (< p).  The point at infinity is (0, 0),
 * which is never on the curve because 3 is not a square mod p.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;

/* ORACLE_MUTATION plants one deliberate mistake (tests/test_oracle_mutations.py
 * builds each variant and checks that the pins reject it).  0 = correct code. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif
#define MUT(n) (ORACLE_MUTATION == (n))

/* ---------------------------------------------------------------- moduli */

typedef struct {
    uint64_t m[4];  /* the modulus, 254 bits */
    uint64_t mu[5]; /* floor(2^512 / m), Barrett constant */
} modulus;

static modulus FP, FR;
static uint64_t MONT_R[4];     /* 2^256 mod p */
static uint64_t MONT_RINV[4];  /* 2^-256 mod p */
static uint64_t COMB[32][256][8]; /* [j * 2^(8w)]G, canonical affine; j = 0 is infinity */
static int g_comb_ready = 0;
static int g_ready = 0;
static pthread_mutex_t g_init_lock = PTHREAD_MUTEX_INITIALIZER;

/* p and r of BN254, written out from their defining polynomials in
 * u = 4965661367192848881 (checked by the test-suite against those
 * polynomials and for primality). */
static const uint64_t P_WORDS[4] = {0x3c208c16d87cfd47ULL, 0x97816a916871ca8dULL,
                                    0xb85045b68181585dULL, 0x30644e72e131a029ULL};
static const uint64_t R_WORDS[4] = {0x43e1f593f0000001ULL, 0x2833e84879b97091ULL,
                                    0xb85045b68181585dULL, 0x30644e72e131a029ULL};

/* a >= b on n limbs */
static int geq_n(const uint64_t *a, const uint64_t *b, int n) {
    for (int i = n - 1; i >= 0; i--) {
        if (a[i] != b[i]) return a[i] > b[i];
    }
    return 1;
}

/* a -= b on n limbs, returns borrow */
static uint64_t sub_n(uint64_t *a, const uint64_t *b, int n) {
    uint64_t borrow = 0;
    for (int i = 0; i < n; i++) {
        u128 d = (u128)a[i] - b[i] - borrow;
        a[i] = (uint64_t)d;
        borrow = (uint64_t)(d >> 64) ? 1 : 0;
    }
    return borrow;
}

/* a += b on n limbs, returns carry */
static uint64_t add_n(uint64_t *a, const uint64_t *b, int n) {
    uint64_t carry = 0;
    for (int i = 0; i < n; i++) {
        u128 s = (u128)a[i] + b[i] + carry;
        a[i] = (uint64_t)s;
        carry = (uint64_t)(s >> 64);
    }
    return carry;
}

/* full product of an na-limb and an nb-limb number into na+nb limbs */
static void mul_full(const uint64_t *a, int na, const uint64_t *b, int nb, uint64_t *out) {
    memset(out, 0, sizeof(uint64_t) * (size_t)(na + nb));
    for (int i = 0; i < na; i++) {
        uint64_t carry = 0;
        for (int j = 0; j < nb; j++) {
            u128 t = (u128)a[i] * b[j] + out[i + j] + carry;
            out[i + j] = (uint64_t)t;
            carry = (uint64_t)(t >> 64);
        }
        out[i + nb] = carry;
    }
}

/* mu = floor(2^512 / m) by schoolbook binary long division, one bit at a time. */
static void barrett_setup(modulus *md, const uint64_t *m) {
    memcpy(md->m, m, sizeof md->m);
    uint64_t rem[5] = {0, 0, 0, 0, 0};
    uint64_t q[9] = {0};
    uint64_t mm[5] = {m[0], m[1], m[2], m[3], 0};
    for (int bit = 512; bit >= 0; bit--) {
        /* rem = 2*rem + bit(2^512, bit) */
        uint64_t top = 0;
        for (int i = 0; i < 5; i++) {
            uint64_t nt = rem[i] >> 63;
            rem[i] = (rem[i] << 1) | top;
            top = nt;
        }
        if (bit == 512) rem[0] |= 1;
        if (geq_n(rem, mm, 5)) {
            sub_n(rem, mm, 5);
            q[bit / 64] |= 1ULL << (bit % 64);
        }
    }
    memcpy(md->mu, q, sizeof md->mu); /* the quotient fits in 5 limbs */
}

/* r = x mod m for x < 2^512 (8 limbs): HAC Algorithm 14.42 with b = 2^64, k = 4. */
static void barrett_reduce(const modulus *md, const uint64_t *x, uint64_t *r) {
    const uint64_t *q1 = x + 3;     /* floor(x / b^(k-1)), 5 limbs */
    uint64_t q2[10];
    mul_full(q1, 5, md->mu, 5, q2); /* q1 * mu */
    const uint64_t *q3 = q2 + 5;    /* floor(q2 / b^(k+1)), 5 limbs */
    uint64_t r2full[9];
    mul_full(q3, 5, md->m, 4, r2full);
    uint64_t rr[5] = {x[0], x[1], x[2], x[3], x[4]}; /* x mod b^(k+1) */
    sub_n(rr, r2full, 5);                            /* mod b^(k+1): wraps if negative */
    uint64_t mm[5] = {md->m[0], md->m[1], md->m[2], md->m[3], 0};
    /* HAC bounds the remainder by 3m; for a 254-bit m with b = 2^64, k = 4 the
     * quotient estimate is off by at most one, so the loop runs at most once. */
    if (!MUT(3)) while (geq_n(rr, mm, 5)) sub_n(rr, mm, 5);
    memcpy(r, rr, 4 * sizeof(uint64_t));
}

/* ------------------------------------------------------ field arithmetic */

typedef struct { uint64_t v[4]; } fe;

static int fe_is_zero(const fe *a) { return (a->v[0] | a->v[1] | a->v[2] | a->v[3]) == 0; }
static int fe_eq(const fe *a, const fe *b) { return memcmp(a->v, b->v, sizeof a->v) == 0; }

static void fe_add(const modulus *md, fe *o, const fe *a, const fe *b) {
    uint64_t s[5] = {a->v[0], a->v[1], a->v[2], a->v[3], 0};
    uint64_t bb[5] = {b->v[0], b->v[1], b->v[2], b->v[3], 0};
    add_n(s, bb, 5);
    uint64_t mm[5] = {md->m[0], md->m[1], md->m[2], md->m[3], 0};
    if (geq_n(s, mm, 5)) sub_n(s, mm, 5);
    memcpy(o->v, s, sizeof o->v);
}

static void fe_sub(const modulus *md, fe *o, const fe *a, const fe *b) {
    uint64_t s[4];
    memcpy(s, a->v, sizeof s);
    if (sub_n(s, b->v, 4)) add_n(s, md->m, 4);
    memcpy(o->v, s, sizeof o->v);
}

static void fe_mul(const modulus *md, fe *o, const fe *a, const fe *b) {
    uint64_t t[8];
    mul_full(a->v, 4, b->v, 4, t);
    barrett_reduce(md, t, o->v);
}

/* a^e for a 256-bit exponent, left-to-right square and multiply */
static void fe_pow(const modulus *md, fe *o, const fe *a, const uint64_t *e) {
    fe acc = {{1, 0, 0, 0}};
    for (int bit = 255; bit >= 0; bit--) {
        fe_mul(md, &acc, &acc, &acc);
        if ((e[bit / 64] >> (bit % 64)) & 1) fe_mul(md, &acc, &acc, a);
    }
    *o = acc;
}

/* Fermat: a^(m-2); the modulus is prime.  inv(0) returns 0. */
static void fe_inv(const modulus *md, fe *o, const fe *a) {
    uint64_t e[4];
    memcpy(e, md->m, sizeof e);
    uint64_t two[4] = {2, 0, 0, 0};
    sub_n(e, two, 4);
    fe_pow(md, o, a, e);
}

/* reduce an arbitrary 256-bit integer into [0, m) */
static void fe_from_u256(const modulus *md, fe *o, const uint64_t *x) {
    uint64_t t[8] = {x[0], x[1], x[2], x[3], 0, 0, 0, 0};
    barrett_reduce(md, t, o->v);
}

/* ------------------------------------------------------- curve arithmetic */

/* Jacobian (X, Y, Z): x = X/Z^2, y = Y/Z^3; Z = 0 is the point at infinity. */
typedef struct { fe X, Y, Z; } jac;
typedef struct { fe x, y; int inf; } aff;

static void jac_set_inf(jac *p) { memset(p, 0, sizeof *p); }
static int jac_is_inf(const jac *p) { return fe_is_zero(&p->Z); }

static void jac_from_aff(jac *o, const aff *a) {
    if (a->inf) { jac_set_inf(o); return; }
    o->X = a->x;
    o->Y = a->y;
    memset(&o->Z, 0, sizeof o->Z);
    o->Z.v[0] = 1;
}

static void jac_to_aff(aff *o, const jac *p) {
    if (jac_is_inf(p)) { memset(o, 0, sizeof *o); o->inf = 1; return; }
    fe zi, zi2, zi3;
    fe_inv(&FP, &zi, &p->Z);
    fe_mul(&FP, &zi2, &zi, &zi);
    fe_mul(&FP, &zi3, &zi2, &zi);
    fe_mul(&FP, &o->x, &p->X, &zi2);
    fe_mul(&FP, &o->y, &p->Y, &zi3);
    o->inf = 0;
}

/* Doubling for a = 0 (Hankerson-Menezes-Vanstone, Guide to ECC, section 3.2.2):
 * S = 4 X Y^2, M = 3 X^2, X' = M^2 - 2S, Y' = M (S - X') - 8 Y^4, Z' = 2 Y Z. */
static void jac_double(jac *o, const jac *p) {
    if (jac_is_inf(p) || fe_is_zero(&p->Y)) { jac_set_inf(o); return; }
    fe y2, s, m, x2, t, y4, xo, yo, zo;
    fe_mul(&FP, &y2, &p->Y, &p->Y);
    fe_mul(&FP, &s, &p->X, &y2);
    fe_add(&FP, &s, &s, &s);
    fe_add(&FP, &s, &s, &s);            /* S = 4 X Y^2 */
    fe_mul(&FP, &x2, &p->X, &p->X);
    fe_add(&FP, &m, &x2, &x2);
    fe_add(&FP, &m, &m, &x2);           /* M = 3 X^2 */
    fe_mul(&FP, &xo, &m, &m);
    fe_sub(&FP, &xo, &xo, &s);
    fe_sub(&FP, &xo, &xo, &s);          /* X' = M^2 - 2S */
    fe_mul(&FP, &y4, &y2, &y2);
    fe_add(&FP, &y4, &y4, &y4);
    fe_add(&FP, &y4, &y4, &y4);
    fe_add(&FP, &y4, &y4, &y4);         /* 8 Y^4 */
    fe_sub(&FP, &t, &s, &xo);
    fe_mul(&FP, &yo, &m, &t);
    if (!MUT(1)) fe_sub(&FP, &yo, &yo, &y4); /* Y' = M (S - X') - 8 Y^4 */
    fe_mul(&FP, &zo, &p->Y, &p->Z);
    fe_add(&FP, &zo, &zo, &zo);         /* Z' = 2 Y Z */
    o->X = xo; o->Y = yo; o->Z = zo;
}

/* General addition: U1 = X1 Z2^2, U2 = X2 Z1^2, S1 = Y1 Z2^3, S2 = Y2 Z1^3,
 * H = U2 - U1, R = S2 - S1, X3 = R^2 - H^3 - 2 U1 H^2,
 * Y3 = R (U1 H^2 - X3) - S1 H^3, Z3 = H Z1 Z2.  Equal inputs double, opposite
 * inputs give infinity. */
static void jac_add(jac *o, const jac *p, const jac *q) {
    if (jac_is_inf(p)) { *o = *q; return; }
    if (jac_is_inf(q)) { *o = *p; return; }
    fe z1s, z2s, u1, u2, s1, s2, t;
    fe_mul(&FP, &z1s, &p->Z, &p->Z);
    fe_mul(&FP, &z2s, &q->Z, &q->Z);
    fe_mul(&FP, &u1, &p->X, &z2s);
    fe_mul(&FP, &u2, &q->X, &z1s);
    fe_mul(&FP, &t, &q->Z, &z2s);
    fe_mul(&FP, &s1, &p->Y, &t);
    fe_mul(&FP, &t, &p->Z, &z1s);
    fe_mul(&FP, &s2, &q->Y, &t);
    if (fe_eq(&u1, &u2)) {
        if (fe_eq(&s1, &s2) && !MUT(8)) { jac_double(o, p); return; }
        jac_set_inf(o);
        return;
    }
    fe h, r, h2, h3, u1h2, xo, yo, zo;
    fe_sub(&FP, &h, &u2, &u1);
    fe_sub(&FP, &r, &s2, &s1);
    fe_mul(&FP, &h2, &h, &h);
    fe_mul(&FP, &h3, &h2, &h);
    fe_mul(&FP, &u1h2, &u1, &h2);
    fe_mul(&FP, &xo, &r, &r);
    fe_sub(&FP, &xo, &xo, &h3);
    fe_sub(&FP, &xo, &xo, &u1h2);
    fe_sub(&FP, &xo, &xo, &u1h2);
    fe_sub(&FP, &t, &u1h2, &xo);
    fe_mul(&FP, &yo, &r, &t);
    fe_mul(&FP, &t, &s1, &h3);
    if (MUT(2)) fe_add(&FP, &yo, &yo, &t);
    else fe_sub(&FP, &yo, &yo, &t);
    fe_mul(&FP, &zo, &h, &p->Z);
    fe_mul(&FP, &zo, &zo, &q->Z);
    o->X = xo; o->Y = yo; o->Z = zo;
}

/* [k]P, left to right over all 256 bits of k. */
static void jac_scalar_mul(jac *o, const jac *p, const uint64_t *k) {
    jac acc;
    jac_set_inf(&acc);
    for (int bit = MUT(4) ? 254 : 255; bit >= 0; bit--) {
        jac_double(&acc, &acc);
        if ((k[bit / 64] >> (bit % 64)) & 1) jac_add(&acc, &acc, p);
    }
    *o = acc;
}

static void aff_load(aff *a, const uint64_t *w) {
    memcpy(a->x.v, w, 32);
    memcpy(a->y.v, w + 4, 32);
    a->inf = fe_is_zero(&a->x) && fe_is_zero(&a->y);
}

static void aff_store(uint64_t *w, const aff *a) {
    if (a->inf) { memset(w, 0, 64); return; }
    memcpy(w, a->x.v, 32);
    memcpy(w + 4, a->y.v, 32);
}

/* ------------------------------------------------------------------ setup */

static void setup_locked(void) {
    barrett_setup(&FP, P_WORDS);
    barrett_setup(&FR, R_WORDS);
    /* 2^256 mod p: reduce the 8-limb integer 2^256 */
    uint64_t t[8] = {0, 0, 0, 0, 1, 0, 0, 0};
    barrett_reduce(&FP, t, MONT_R);
    fe rr, ri;
    memcpy(rr.v, MONT_R, 32);
    fe_inv(&FP, &ri, &rr);
    memcpy(MONT_RINV, ri.v, 32);
}

int oracle_init(void) {
    pthread_mutex_lock(&g_init_lock);
    if (!g_ready) { setup_locked(); g_ready = 1; }
    pthread_mutex_unlock(&g_init_lock);
    return 0;
}


/* Comb table for fixed-base multiples of G = (1, 2): since
 * k = sum_w byte_w(k) * 2^(8w), [k]G = sum_w COMB[w][byte_w(k)]. */
static void comb_setup_locked(void) {
    jac base;
    memset(&base, 0, sizeof base);
    base.X.v[0] = 1; base.Y.v[0] = 2; base.Z.v[0] = 1;   /* [2^(8w)]G, w = 0 */
    for (int w = 0; w < 32; w++) {
        jac acc;
        jac_set_inf(&acc);
        memset(COMB[w][0], 0, 64);
        for (int j = 1; j < 256; j++) {
            aff a;
            jac_add(&acc, &acc, &base);                     /* [j * 2^(8w)]G */
            jac_to_aff(&a, &acc);
            aff_store(COMB[w][j], &a);
        }
        for (int d = 0; d < 8; d++) jac_double(&base, &base);
    }
}

static void comb_init(void) {
    oracle_init();
    pthread_mutex_lock(&g_init_lock);
    if (!g_comb_ready) { comb_setup_locked(); g_comb_ready = 1; }
    pthread_mutex_unlock(&g_init_lock);
}

/* ---------------------------------------------------------- parallel map */

typedef struct {
    size_t begin, end;
    const uint64_t *a, *b;
    uint64_t *out;
    jac partial;
} task;

static int run_threads(void *(*fn)(void *), task *tasks, int nthreads) {
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) return -1;
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; t++) {
        if (pthread_create(&tid[t], NULL, fn, &tasks[t]) != 0) { rc = -1; break; }
        started++;
    }
    for (int t = 0; t < started; t++) pthread_join(tid[t], NULL);
    free(tid);
    return rc;
}

static int clamp_threads(int nthreads, size_t n) {
    if (nthreads < 1) nthreads = 1;
    if ((size_t)nthreads > n) nthreads = (int)(n ? n : 1);
    return nthreads;
}

/* ------------------------------------------------------------- exported */

/* out_i = [k_i]G as canonical affine, summing one comb entry per byte of k_i. */
static void *gen_worker(void *arg) {
    task *tk = (task *)arg;
    for (size_t i = tk->begin; i < tk->end; i++) {
        const uint64_t *k = tk->a + 4 * i;
        jac acc;
        jac_set_inf(&acc);
        for (int w = 0; w < 32; w++) {
            int ww = MUT(7) ? (w + 1) % 32 : w;
            unsigned byte = (unsigned)((k[ww / 8] >> (8 * (ww % 8))) & 0xFF);
            if (byte) {
                aff t;
                jac tj;
                aff_load(&t, COMB[w][byte]);
                jac_from_aff(&tj, &t);
                jac_add(&acc, &acc, &tj);
            }
        }
        aff a;
        jac_to_aff(&a, &acc);
        aff_store(tk->out + 8 * i, &a);
    }
    return NULL;
}

int oracle_g1_generator_multiples(const uint64_t *k, size_t n, uint64_t *out, int nthreads) {
    comb_init();
    if (n == 0) return 0;
    if (!k || !out) return -1;
    nthreads = clamp_threads(nthreads, n);
    task *tasks = (task *)calloc((size_t)nthreads, sizeof(task));
    if (!tasks) return -1;
    for (int t = 0; t < nthreads; t++) {
        tasks[t].begin = n * (size_t)t / (size_t)nthreads;
        tasks[t].end = n * (size_t)(t + 1) / (size_t)nthreads;
        tasks[t].a = k;
        tasks[t].out = out;
    }
    int rc = run_threads(gen_worker, tasks, nthreads);
    free(tasks);
    return rc;
}

/* partial_t = sum over its range of [k_i]P_i (one scalar multiplication per term) */
static void *msm_worker(void *arg) {
    task *tk = (task *)arg;
    jac acc;
    jac_set_inf(&acc);
    for (size_t i = tk->begin; i < tk->end - (MUT(5) && tk->end > tk->begin ? 1 : 0); i++) {
        aff p;
        jac pj, term;
        aff_load(&p, tk->a + 8 * i);
        jac_from_aff(&pj, &p);
        jac_scalar_mul(&term, &pj, tk->b + 4 * i);
        jac_add(&acc, &acc, &term);
    }
    tk->partial = acc;
    return NULL;
}

/* Q = sum_i [k_i] P_i; points canonical affine (8 u64 each), scalars 4 u64 each
 * (any 256-bit value), out canonical affine (8 u64; (0,0) = infinity). */
int oracle_msm(const uint64_t *pts, const uint64_t *scalars, size_t n, uint64_t *out, int nthreads) {
    oracle_init();
    if (!out) return -1;
    if (n == 0) { memset(out, 0, 64); return 0; }
    if (!pts || !scalars) return -1;
    nthreads = clamp_threads(nthreads, n);
    task *tasks = (task *)calloc((size_t)nthreads, sizeof(task));
    if (!tasks) return -1;
    for (int t = 0; t < nthreads; t++) {
        tasks[t].begin = n * (size_t)t / (size_t)nthreads;
        tasks[t].end = n * (size_t)(t + 1) / (size_t)nthreads;
        tasks[t].a = pts;
        tasks[t].b = scalars;
    }
    int rc = run_threads(msm_worker, tasks, nthreads);
    jac total;
    jac_set_inf(&total);
    for (int t = 0; t < nthreads; t++) jac_add(&total, &total, &tasks[t].partial);
    free(tasks);
    aff a;
    jac_to_aff(&a, &total);
    aff_store(out, &a);
    return rc;
}

/* x -> x * 2^256 mod p (Montgomery encoding) for nelem field elements */
int oracle_mont_encode(const uint64_t *in, size_t nelem, uint64_t *out) {
    oracle_init();
    fe r;
    memcpy(r.v, MONT_R, 32);
    for (size_t i = 0; i < nelem; i++) {
        fe a, o;
        fe_from_u256(&FP, &a, in + 4 * i);
        fe_mul(&FP, &o, &a, &r);
        memcpy(out + 4 * i, o.v, 32);
    }
    return 0;
}

/* x~ -> x~ * 2^-256 mod p (Montgomery decoding) */
int oracle_mont_decode(const uint64_t *in, size_t nelem, uint64_t *out) {
    oracle_init();
    fe ri;
    memcpy(ri.v, MUT(6) ? MONT_R : MONT_RINV, 32);
    for (size_t i = 0; i < nelem; i++) {
        fe a, o;
        fe_from_u256(&FP, &a, in + 4 * i);
        fe_mul(&FP, &o, &a, &ri);
        memcpy(out + 4 * i, o.v, 32);
    }
    return 0;
}

/* Jacobian point with Montgomery-encoded X, Y, Z (12 u64) -> canonical affine (8 u64) */
int oracle_jacobian_mont_to_affine(const uint64_t *jm, uint64_t *out) {
    oracle_init();
    uint64_t dec[12];
    oracle_mont_decode(jm, 3, dec);
    jac p;
    memcpy(p.X.v, dec, 32);
    memcpy(p.Y.v, dec + 4, 32);
    memcpy(p.Z.v, dec + 8, 32);
    aff a;
    jac_to_aff(&a, &p);
    aff_store(out, &a);
    return 0;
}

int oracle_g1_add(const uint64_t *a, const uint64_t *b, uint64_t *out) {
    oracle_init();
    aff pa, pb, r;
    jac ja, jb, jr;
    aff_load(&pa, a);
    aff_load(&pb, b);
    jac_from_aff(&ja, &pa);
    jac_from_aff(&jb, &pb);
    jac_add(&jr, &ja, &jb);
    jac_to_aff(&r, &jr);
    aff_store(out, &r);
    return 0;
}

int oracle_g1_scalar_mul(const uint64_t *pt, const uint64_t *k, uint64_t *out) {
    oracle_init();
    aff p, r;
    jac jp, jr;
    aff_load(&p, pt);
    jac_from_aff(&jp, &p);
    jac_scalar_mul(&jr, &jp, k);
    jac_to_aff(&r, &jr);
    aff_store(out, &r);
    return 0;
}

/* 1 if the point is infinity or satisfies y^2 = x^3 + 3 with canonical coordinates */
int oracle_g1_is_on_curve(const uint64_t *pt) {
    oracle_init();
    aff p;
    aff_load(&p, pt);
    if (MUT(9)) return 1;
    if (p.inf) return 1;
    if (!MUT(10) && (geq_n(p.x.v, FP.m, 4) || geq_n(p.y.v, FP.m, 4))) return 0;
    fe y2, x3, three = {{3, 0, 0, 0}};
    fe_mul(&FP, &y2, &p.y, &p.y);
    fe_mul(&FP, &x3, &p.x, &p.x);
    fe_mul(&FP, &x3, &x3, &p.x);
    fe_add(&FP, &x3, &x3, &three);
    return fe_eq(&y2, &x3);
}

/* sum_i a_i * b_i mod r, both operands any 256-bit integers */
int oracle_scalar_dot_mod_r(const uint64_t *a, const uint64_t *b, size_t n, uint64_t *out) {
    oracle_init();
    fe acc = {{0, 0, 0, 0}};
    for (size_t i = 0; i < n; i++) {
        fe x, y, t;
        fe_from_u256(&FR, &x, a + 4 * i);
        fe_from_u256(&FR, &y, b + 4 * i);
        fe_mul(&FR, &t, &x, &y);
        fe_add(&FR, &acc, &acc, &t);
    }
    memcpy(out, acc.v, 32);
    return 0;
}

/* field helpers exposed for the pins: o = a*b mod p, o = a^-1 mod p */
int oracle_fp_mul(const uint64_t *a, const uint64_t *b, uint64_t *out) {
    oracle_init();
    fe x, y, o;
    fe_from_u256(&FP, &x, a);
    fe_from_u256(&FP, &y, b);
    fe_mul(&FP, &o, &x, &y);
    memcpy(out, o.v, 32);
    return 0;
}

int oracle_fp_inv(const uint64_t *a, uint64_t *out) {
    oracle_init();
    fe x, o;
    fe_from_u256(&FP, &x, a);
    fe_inv(&FP, &o, &x);
    memcpy(out, o.v, 32);
    return 0;
}
