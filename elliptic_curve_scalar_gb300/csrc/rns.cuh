// rns.cuh -- F_p arithmetic in a residue number system (RNS), spread over the
// 10 lanes of a warp group, for the latency-bound chains of the MSM.
//
// A single-lane Montgomery product (fq.cuh) issues 264 multiply-pipe slots
// from one warp, so a chain of dependent products -- the window
// combination's ~115 doublings -- runs at one product per ~870 cycles however
// many lanes wait.  In an RNS an integer is held as its residues modulo
// pairwise coprime moduli and a product is one 32-bit product per residue;
// Montgomery's reduction becomes two base extensions, each a 9-term dot
// product per lane over values gathered by shuffles (Bajard, Didier and
// Kornerup, "An RNS Montgomery modular multiplication algorithm", IEEE Trans.
// Computers 47(7), 1998; the exact second extension with a redundant modulus
// after Shenoy and Kumaresan, IEEE Trans. Computers 38(2), 1989).
//
// Layout.  Base B = 9 primes m_j = 2^32 - c_j, base B' = 9 more, redundant
// modulus 2^32 (rns_consts.cuh, written by gen_rns.py; every c_j < 2^11).  A
// group is 10 consecutive lanes; lane j < 9 holds the residue mod m_j (slot
// a) and mod m'_j (slot b), lane 9 the residue mod 2^32 in both slots.  The B
// residues are stored times lambda_j, a square root of the product's first
// constant c1_j = -p^-1 (M/m_j)^-1 mod m_j, so that x' y' = x y c1_j is the
// product's first step in one multiplication (gen_rns.py picks B so that
// every c1_j is a square).  A warp holds three groups (lanes 0-9, 10-19,
// 20-29) that work on three products at once; lanes 30 and 31 follow along on
// a copy of group 0's channels and their results are never used.  Every
// function is called by all 32 lanes of a converged warp.
//
// Residues are lazy: any 32-bit representative of the residue, reduced to
// the canonical one in [0, m) only where a comparison or the CRT needs it.
// Folding uses 2^32 = c mod m; for the redundant lane c = 0 and every fold is
// the identity, so the same instructions give exact arithmetic mod 2^32.
//
// Values.  An RNS value is a non-negative integer X, below a small multiple
// of p, standing for the field element X M^-1 mod p (M = prod of B): the
// RNS Montgomery domain, in which mm(X, Y) = X Y M^-1 represents the product.
// With lazy residues the first extension's q may exceed q mod M by less than
// 18 M, so mm returns an integer below (18 + K_x K_y p / M) p < 20 p for
// inputs below K_x p and K_y p with K_x K_y < 2^30 (M > 2^287, p < 2^254).
// Subtraction adds a multiple of p first, X + k p - Y with k p above Y's
// bound, so values stay non-negative; every call site states its bounds.
#pragma once
#include <stdint.h>

#include "fq.cuh"
#include "rns_consts.cuh"

namespace rns {

// constants of one lane, in the order gen_rns.py writes them
struct Lane {
    uint32_t ca, cb, ma, mb, pb, minv, minvc2, mpa, mpinv, pinv, pa, crt, cin_a, cin_b, cout_a, cout_b;
    uint32_t e1[9], e2[9], pow_a[8], pow_b[8];
};

struct Ctx {
    Lane k;
    int j;     // lane within the group (0..9)
    int base;  // first lane of the group
    int g;     // group 0..2 (3 for lanes 30 and 31)
};

__device__ __forceinline__ Ctx make_ctx() {
    Ctx C;
    const int lane = threadIdx.x & 31;
    C.g = lane / 10;
    C.j = lane % 10;
    C.base = C.g < 3 ? C.g * 10 : 0;
    const uint32_t* src = kLane[C.j];
    uint32_t* dst = reinterpret_cast<uint32_t*>(&C.k);
#pragma unroll
    for (int i = 0; i < 50; i++) {
        dst[i] = __ldg(src + i);
        // keep the constant in its register: without this the compiler may
        // reload it from memory inside the latency-bound chains
        asm volatile("" : "+r"(dst[i]));
    }
    return C;
}

// one lane's two residues of a value
struct rv {
    uint32_t a, b;
};

// A 32-bit representative of v mod m, m = 2^32 - c, for v < 2^48: fold the
// high word in twice (2^32 = c mod m); the second fold's high word is 0 or 1.
__device__ __forceinline__ uint32_t fold(uint64_t v, uint32_t c) {
    const uint64_t w = (v >> 32) * c + (uint32_t)v;  // < 2^27 + 2^32
    return (uint32_t)w + (uint32_t)(w >> 32) * c;    // high word 1 leaves a low word below 2^27
}
// x y mod m, lazily
__device__ __forceinline__ uint32_t mulmod(uint32_t x, uint32_t y, uint32_t c) {
    const uint64_t t = (uint64_t)x * y;
    return fold((t >> 32) * c + (uint32_t)t, c);  // < 2^43 + 2^32
}
// the canonical residue in [0, m) of a lazy one
__device__ __forceinline__ uint32_t canon(uint32_t x, uint32_t c) {
    const uint64_t t = (uint64_t)x + c;
    return (t >> 32) ? (uint32_t)t : x;
}
// sum_i x_i e_i mod m, lazily: each product folded once, the folds summed in
// a balanced tree, the sum folded
template <int N>
__device__ __forceinline__ uint32_t dot(const uint32_t (&x)[N], const uint32_t* e, uint32_t c) {
    uint64_t u[N];
#pragma unroll
    for (int i = 0; i < N; i++) {
        const uint64_t t = (uint64_t)x[i] * e[i];
        u[i] = (t >> 32) * c + (uint32_t)t;  // < 2^43 + 2^32
    }
#pragma unroll
    for (int w = 1; w < N; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < N; i += 2 * w) u[i] += u[i + w];
    return fold(u[0], c);  // < 9 (2^43 + 2^32) < 2^47
}

// x + y
__device__ __forceinline__ rv add(const Ctx& C, rv x, rv y) {
    return {fold((uint64_t)x.a + y.a, C.k.ca), fold((uint64_t)x.b + y.b, C.k.cb)};
}
// k p as an RNS integer (canonical residues), for sub
__device__ __forceinline__ rv kp(const Ctx& C, uint32_t k) {
    return {canon(mulmod(C.k.pa, k, C.k.ca), C.k.ca), canon(mulmod(C.k.pb, k, C.k.cb), C.k.cb)};
}
// x + kp - s y for a small s (kp from kp(), above s times y's bound): a lazy
// residue is below 2^32 <= 2m, so the offset 2 s m per channel keeps the
// 64-bit sum non-negative; m is 2^32 in the redundant lane, where the offset
// vanishes mod 2^32
__device__ __forceinline__ rv sub(const Ctx& C, rv x, rv y, rv kp, uint32_t s = 1) {
    const uint64_t ma = C.k.ma ? C.k.ma : (1ull << 32), mb = C.k.mb ? C.k.mb : (1ull << 32);
    return {fold((uint64_t)x.a + kp.a + 2 * s * ma - (uint64_t)s * y.a, C.k.ca),
            fold((uint64_t)x.b + kp.b + 2 * s * mb - (uint64_t)s * y.b, C.k.cb)};
}
// x times a small integer k (the represented element times k)
__device__ __forceinline__ rv mul_small(const Ctx& C, rv x, uint32_t k) {
    return {fold((uint64_t)x.a * k, C.k.ca), fold((uint64_t)x.b * k, C.k.cb)};
}

// the residues of this lane's group for value v, from group `from` (the same channel)
__device__ __forceinline__ rv from_group(const Ctx& C, rv v, int from) {
    const int src = from * 10 + C.j;
    return {__shfl_sync(0xffffffffu, v.a, src), __shfl_sync(0xffffffffu, v.b, src)};
}

// X Y M^-1 mod p (lazily, see the file comment).
//  1. in B: xi_j = x'_j y'_j = t_j c1_j (the scaled residues), so that
//     q = sum xi_j M/m_j (mod M) makes t + q p divisible by M;
//  2. fast extension of q to B' and 2^32 (no correction: with lazy xi, q may
//     exceed a multiple of M below 18 M, which only adds a multiple of p
//     below 18 p to r);
//  3. r = (t + q p) / M in B' and 2^32, and xi'_j = r (M'/m'_j)^-1 from the
//     same sum t + q p;
//  4. exact extension of r back to B: r = sum xi'_j M'/m'_j - beta M' with
//     beta < 18 found exactly in the redundant channel:
//     beta = (sum xi'_j (M'/m'_j) - r) M'^-1 mod 2^32.
__device__ __forceinline__ rv mm(const Ctx& C, rv x, rv y) {
    const uint32_t xi = mulmod(x.a, y.a, C.k.ca);
    const uint32_t tb = mulmod(x.b, y.b, C.k.cb);
    uint32_t v[9];
#pragma unroll
    for (int i = 0; i < 9; i++) v[i] = __shfl_sync(0xffffffffu, xi, C.base + i);
    const uint32_t q = dot<9>(v, C.k.e1, C.k.cb);
    const uint64_t tq = (uint64_t)q * C.k.pb + tb;
    const uint32_t s1 = fold((tq >> 32) * C.k.cb + (uint32_t)tq, C.k.cb);
    const uint32_t rb = mulmod(s1, C.k.minv, C.k.cb);
    const uint32_t xi2 = mulmod(s1, C.k.minvc2, C.k.cb);
#pragma unroll
    for (int i = 0; i < 9; i++) v[i] = __shfl_sync(0xffffffffu, xi2, C.base + i);
    const uint32_t s = dot<9>(v, C.k.e2, C.k.ca);
    // in the redundant lane s and rb are exact mod 2^32
    const uint32_t beta = __shfl_sync(0xffffffffu, (s - rb) * C.k.mpinv, C.base + 9);
    const uint64_t ma = C.k.ma ? C.k.ma : (1ull << 32);
    return {fold((uint64_t)s + 18 * ma - (uint64_t)beta * C.k.mpa, C.k.ca), rb};
}

// Three products at once, one per group: group g computes x_g y_g; every
// group receives all three.
__device__ __forceinline__ void mm3(const Ctx& C, rv x0, rv y0, rv x1, rv y1, rv x2, rv y2, rv& p0, rv& p1, rv& p2) {
    const rv x = C.g == 0 ? x0 : C.g == 1 ? x1 : C.g == 2 ? x2 : x0;
    const rv y = C.g == 0 ? y0 : C.g == 1 ? y1 : C.g == 2 ? y2 : y0;
    const rv p = mm(C, x, y);
    p0 = from_group(C, p, 0);
    p1 = from_group(C, p, 1);
    p2 = from_group(C, p, 2);
}

// the residues of a positional integer x < 2^256 (8 words), before the domain change
__device__ __forceinline__ rv residues(const Ctx& C, const fq::fe& x) {
    return {dot<8>(x.v, C.k.pow_a, C.k.ca), dot<8>(x.v, C.k.pow_b, C.k.cb)};
}
// into the RNS Montgomery domain from positional Montgomery form x~ = x R mod p:
// mm(x~, M^2 R^-1 mod p) = x M mod p (below 20 p)
__device__ __forceinline__ rv cin(const Ctx& C) { return {C.k.cin_a, C.k.cin_b}; }
// out of it: mm(X, R mod p) = x R mod p, then to_positional
__device__ __forceinline__ rv cout(const Ctx& C) { return {C.k.cout_a, C.k.cout_b}; }

// The positional integer of an RNS value Y < 32 p, reduced mod p (8 words,
// every lane the same): Y = sum_j xi_j M/m_j - alpha M with xi_j = y_j
// (M/m_j)^-1 mod m_j (canonical) and alpha < 9 exact from the redundant channel.
__device__ __forceinline__ fq::fe to_positional(const Ctx& C, rv y) {
    const uint32_t xi = canon(mulmod(y.a, C.k.crt, C.k.ca), C.k.ca);
    uint32_t v[9];
#pragma unroll
    for (int i = 0; i < 9; i++) v[i] = __shfl_sync(0xffffffffu, xi, C.base + i);
    // alpha = (sum xi_j (M/m_j mod 2^32) - y) M^-1 mod 2^32, in lane 9 (whose
    // e1 row holds M/m_j mod 2^32 and minv M^-1 mod 2^32)
    uint32_t sr = 0;
#pragma unroll
    for (int i = 0; i < 9; i++) sr += v[i] * C.k.e1[i];
    const uint32_t alpha = __shfl_sync(0xffffffffu, (sr - y.b) * C.k.minv, C.base + 9);
    // T = sum_j xi_j (M/m_j) - alpha M in 10 words (the sum is below 9 M < 2^292)
    uint32_t t[10];
#pragma unroll
    for (int w = 0; w < 10; w++) t[w] = 0;
#pragma unroll
    for (int i = 0; i < 9; i++) {
        uint32_t carry = 0;
#pragma unroll
        for (int w = 0; w < 10; w++) {
            const uint64_t s = (uint64_t)v[i] * kMdiv[i][w] + t[w] + carry;
            t[w] = (uint32_t)s;
            carry = (uint32_t)(s >> 32);
        }
    }
    {
        uint32_t borrow = 0;
#pragma unroll
        for (int w = 0; w < 10; w++) {
            const uint64_t s = (uint64_t)alpha * kM[w] + borrow;
            const uint32_t sub = (uint32_t)s;
            borrow = (uint32_t)(s >> 32) + (t[w] < sub);
            t[w] -= sub;
        }
    }
    // now t < 32 p < 2^259: subtract 16p, 8p, 4p, 2p, p where they fit
#pragma unroll
    for (int k = 0; k < 5; k++) {
        uint32_t d[9], br = 0;
#pragma unroll
        for (int w = 0; w < 9; w++) {
            const uint64_t s = (uint64_t)t[w] - kPmul[k][w] - br;
            d[w] = (uint32_t)s;
            br = (uint32_t)(s >> 32) & 1u;
        }
        if (!br) {
#pragma unroll
            for (int w = 0; w < 9; w++) t[w] = d[w];
        }
    }
    fq::fe r;
#pragma unroll
    for (int w = 0; w < 8; w++) r.v[w] = t[w];
    return r;
}

// Is the represented element zero, for a value below bound * p (bound below
// 2^31)?  Y = X p^-1 mod M in B: if X = k p with k < bound every residue of Y
// is k; otherwise all nine residues equal to one small k would make Y = k by
// the CRT, i.e. X = k p (mod M) with both sides below M, a contradiction.
// Each group answers for its own value.
__device__ __forceinline__ bool is_zero(const Ctx& C, rv x, uint32_t bound) {
    const uint32_t y = canon(mulmod(x.a, C.k.pinv, C.k.ca), C.k.ca);
    const uint32_t y0 = __shfl_sync(0xffffffffu, y, C.base);
    const bool ok = C.j == 9 || (y == y0 && y0 < bound);
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    return ((bal >> C.base) & 0x3FFu) == 0x3FFu;
}

}  // namespace rns
