// glv.cuh -- the BN254 G1 endomorphism and the scalar split it allows.
//
// BN254 has j-invariant 0 (a = 0) and p = 1 mod 3, so Fp holds a primitive
// cube root of unity beta and phi(x, y) = (beta x, y) maps the curve to itself.
// On G1 (prime order r, r = 1 mod 3) phi acts as multiplication by a cube root
// of unity lambda mod r: phi(P) = [lambda] P.  The pair (beta, lambda) below is
// the matching one; the other choice of beta belongs to lambda^2.  This is the
// method of Gallant, Lambert and Vanstone ("Faster point multiplication on
// elliptic curves with efficient endomorphisms", CRYPTO 2001), used here to
// turn an MSM of n terms with 254-bit scalars into one of 2n terms with
// 127-bit scalars: k P = k1 P + k2 phi(P) with k = k1 + lambda k2 (mod r).
//
// The split takes the short lattice basis v1 = (a1, b1), v2 = (a2, b2) of
// {(x, y) : x + lambda y = 0 mod r}, found by the extended Euclidean
// algorithm on (r, lambda) as the GLV paper does (a1 b2 - a2 b1 = r), and
// rounds (k, 0) = x1 v1 + x2 v2 with x1 = k b2 / r, x2 = -k b1 / r to the
// integers c_i = floor(k g_i / 2^256), where g1 = round(b2 2^256 / r) and
// g2 = round(-b1 2^256 / r).  The rounding error
// |x_i - c_i| stays below 1 + 2^-3 for k < r, so
//   k1 = k - c1 a1 - c2 a2,   k2 = -c1 b1 - c2 b2
// satisfy |k_i| < 1.125 (a1 + a2) < 2^127 (a1 + a2 = |b1| + b2 ~ 2^126.8).
// Because |k_i| < 2^127, both are recovered exactly from their residues
// mod 2^128 (bit 127 is the sign), which is all the arithmetic computes.
#pragma once
#include <stdint.h>

// little-endian 32-bit limbs
#define GLV_BETA_MONT 0xd782e155u, 0x71930c11u, 0xffbe3323u, 0xa6bb947cu, 0xd4741444u, 0xaa303344u, 0x26594943u, 0x2c3b3f0du
#define GLV_LAMBDA 0xb99c90ddu, 0x8b17ea66u, 0x8d8daaa7u, 0x5bfc4108u, 0x41a91758u, 0xb3c4d79du, 0u, 0u
#define GLV_G1 0xc7e0b3d7u, 0xd91d232eu, 0x00000002u
#define GLV_G2 0x391eb18eu, 0x7a7bd9d4u, 0xa773d2cfu, 0x4ccef014u, 0x00000002u
#define GLV_A1 0x94d213e3u, 0x89d32568u
#define GLV_A2 0x1221250bu, 0x0be4e154u, 0xeeb859fdu, 0x6f4d8248u
#define GLV_B1_ABS 0x7d4f1128u, 0x8211bbebu, 0xeeb859fcu, 0x6f4d8248u  // b1 < 0
#define GLV_B2 0x94d213e3u, 0x89d32568u

namespace glv {

// o = (a b) mod 2^(32 NO), schoolbook with 64-bit row accumulation
template <int NA, int NB, int NO>
__host__ __device__ __forceinline__ void mul_trunc(const uint32_t (&a)[NA], const uint32_t (&b)[NB],
                                                   uint32_t (&o)[NO]) {
#pragma unroll
    for (int i = 0; i < NO; i++) o[i] = 0;
#pragma unroll
    for (int i = 0; i < NA; i++) {
        uint64_t carry = 0;
#pragma unroll
        for (int j = 0; j < NB; j++) {
            if (i + j < NO) {
                uint64_t t = (uint64_t)a[i] * b[j] + o[i + j] + carry;
                o[i + j] = (uint32_t)t;
                carry = t >> 32;
            }
        }
        if (i + NB < NO) o[i + NB] = (uint32_t)carry;
    }
}

// a -= b mod 2^128
__host__ __device__ __forceinline__ void sub128(uint32_t (&a)[4], const uint32_t (&b)[4]) {
    uint64_t borrow = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint64_t t = (uint64_t)a[i] - b[i] - borrow;
        a[i] = (uint32_t)t;
        borrow = (t >> 32) & 1;
    }
}

// |a| for a 128-bit two's-complement value; returns 1 if a was negative
__host__ __device__ __forceinline__ uint32_t abs128(uint32_t (&a)[4]) {
    const uint32_t neg = a[3] >> 31;
    if (neg) {
        uint64_t carry = 1;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint64_t t = (uint64_t)(~a[i]) + carry;
            a[i] = (uint32_t)t;
            carry = t >> 32;
        }
    }
    return neg;
}

// k (< r, 8 limbs) -> |k1|, |k2| (< 2^127, 4 limbs each) and their signs
__host__ __device__ __forceinline__ void split(const uint32_t (&k)[8], uint32_t (&k1)[4], uint32_t (&k2)[4],
                                               uint32_t& neg1, uint32_t& neg2) {
    const uint32_t g1[3] = {GLV_G1}, g2[5] = {GLV_G2};
    const uint32_t a1[2] = {GLV_A1}, a2[4] = {GLV_A2}, b1[4] = {GLV_B1_ABS}, b2[2] = {GLV_B2};
    uint32_t w1[11], w2[13];
    mul_trunc(k, g1, w1);
    mul_trunc(k, g2, w2);
    const uint32_t c1[2] = {w1[8], w1[9]};                 // c1 < 2^64
    const uint32_t c2[4] = {w2[8], w2[9], w2[10], w2[11]};  // c2 < 2^128
    uint32_t t[4];
    // k1 = k - c1 a1 - c2 a2
#pragma unroll
    for (int i = 0; i < 4; i++) k1[i] = k[i];
    mul_trunc(c1, a1, t);
    sub128(k1, t);
    mul_trunc(c2, a2, t);
    sub128(k1, t);
    // k2 = c1 |b1| - c2 b2
    mul_trunc(c1, b1, k2);
    mul_trunc(c2, b2, t);
    sub128(k2, t);
    neg1 = abs128(k1);
    neg2 = abs128(k2);
}

}  // namespace glv
