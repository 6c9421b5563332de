// fq.cuh -- arithmetic in the BN254 base field F_p on sm_103a.
//
// Representation: 8 x 32-bit little-endian limbs in Montgomery form with
// R = 2^256 (x is stored as x*R mod p), always fully reduced (< p), so equality
// and zero tests are plain limb compares.  The pages' kernels use 13-bit limbs
// in f32 lanes for the same "montgomery products" (PR #23520, section "Why not
// split the inverse loop too?", and PR #23738, section "Notes / caveats", which
// names the 13-bit-limb f32 Montgomery math); on this GPU the 32-bit integer
// multiply-add pipe is the natural unit, so the limbs are 32-bit words and each
// partial product is one mad.lo / mad.hi with the carry flag threaded through.
//
// Multiplication is coarsely integrated operand scanning (CIOS): for each
// limb a_i, t += a_i*b, m = t_0 * (-p^-1 mod 2^32), t = (t + m*p) / 2^32.
// Because p < 2^254, t stays below 2p < 2^255 between rounds, so a round never
// carries past limb 8 and limb 8 is zero again after the shift; the result is
// brought below p by one conditional subtraction.  Every carry chain sits in a
// single asm statement so that nothing can clobber the carry flag inside it.
#pragma once
#include <stdint.h>

namespace fq {

// p = 0x30644e72e131a029b85045b68181585d97816a916871ca8d3c208c16d87cfd47
#define FQ_P0 0xd87cfd47u
#define FQ_P1 0x3c208c16u
#define FQ_P2 0x6871ca8du
#define FQ_P3 0x97816a91u
#define FQ_P4 0x8181585du
#define FQ_P5 0xb85045b6u
#define FQ_P6 0xe131a029u
#define FQ_P7 0x30644e72u
// -p^-1 mod 2^32
#define FQ_NP0 0xe4866389u
// R mod p = 2^256 mod p (Montgomery form of 1)
#define FQ_R0 0xc58f0d9du
#define FQ_R1 0xd35d438du
#define FQ_R2 0xf5c70b3du
#define FQ_R3 0x0a78eb28u
#define FQ_R4 0x7879462cu
#define FQ_R5 0x666ea36fu
#define FQ_R6 0x9a07df2fu
#define FQ_R7 0x0e0a77c1u

struct fe {
    uint32_t v[8];
};

__device__ __forceinline__ fe zero() {
    fe r;
#pragma unroll
    for (int i = 0; i < 8; i++) r.v[i] = 0;
    return r;
}

__device__ __forceinline__ fe one() {
    fe r;
    r.v[0] = FQ_R0; r.v[1] = FQ_R1; r.v[2] = FQ_R2; r.v[3] = FQ_R3;
    r.v[4] = FQ_R4; r.v[5] = FQ_R5; r.v[6] = FQ_R6; r.v[7] = FQ_R7;
    return r;
}

__device__ __forceinline__ bool is_zero(const fe& a) {
    return (a.v[0] | a.v[1] | a.v[2] | a.v[3] | a.v[4] | a.v[5] | a.v[6] | a.v[7]) == 0;
}

__device__ __forceinline__ bool eq(const fe& a, const fe& b) {
    uint32_t d = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) d |= a.v[i] ^ b.v[i];
    return d == 0;
}

// t := t - p if t >= p (t < 2p on entry)
__device__ __forceinline__ void reduce_once(fe& t) {
    uint32_t d0, d1, d2, d3, d4, d5, d6, d7, br;
    asm("sub.cc.u32  %0, %9,  %17;\n\t"
        "subc.cc.u32 %1, %10, %18;\n\t"
        "subc.cc.u32 %2, %11, %19;\n\t"
        "subc.cc.u32 %3, %12, %20;\n\t"
        "subc.cc.u32 %4, %13, %21;\n\t"
        "subc.cc.u32 %5, %14, %22;\n\t"
        "subc.cc.u32 %6, %15, %23;\n\t"
        "subc.cc.u32 %7, %16, %24;\n\t"
        "subc.u32    %8, 0, 0;"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3), "=r"(d4), "=r"(d5), "=r"(d6), "=r"(d7), "=r"(br)
        : "r"(t.v[0]), "r"(t.v[1]), "r"(t.v[2]), "r"(t.v[3]), "r"(t.v[4]), "r"(t.v[5]), "r"(t.v[6]), "r"(t.v[7]),
          "n"(FQ_P0), "n"(FQ_P1), "n"(FQ_P2), "n"(FQ_P3), "n"(FQ_P4), "n"(FQ_P5), "n"(FQ_P6), "n"(FQ_P7));
    // br = 0xffffffff when t < p (keep t), 0 when t >= p (take t - p)
    t.v[0] = (t.v[0] & br) | (d0 & ~br);
    t.v[1] = (t.v[1] & br) | (d1 & ~br);
    t.v[2] = (t.v[2] & br) | (d2 & ~br);
    t.v[3] = (t.v[3] & br) | (d3 & ~br);
    t.v[4] = (t.v[4] & br) | (d4 & ~br);
    t.v[5] = (t.v[5] & br) | (d5 & ~br);
    t.v[6] = (t.v[6] & br) | (d6 & ~br);
    t.v[7] = (t.v[7] & br) | (d7 & ~br);
}

__device__ __forceinline__ fe add(const fe& a, const fe& b) {
    fe s;
    asm("add.cc.u32  %0, %8,  %16;\n\t"
        "addc.cc.u32 %1, %9,  %17;\n\t"
        "addc.cc.u32 %2, %10, %18;\n\t"
        "addc.cc.u32 %3, %11, %19;\n\t"
        "addc.cc.u32 %4, %12, %20;\n\t"
        "addc.cc.u32 %5, %13, %21;\n\t"
        "addc.cc.u32 %6, %14, %22;\n\t"
        "addc.u32    %7, %15, %23;"
        : "=r"(s.v[0]), "=r"(s.v[1]), "=r"(s.v[2]), "=r"(s.v[3]), "=r"(s.v[4]), "=r"(s.v[5]), "=r"(s.v[6]), "=r"(s.v[7])
        : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]),
          "r"(b.v[0]), "r"(b.v[1]), "r"(b.v[2]), "r"(b.v[3]), "r"(b.v[4]), "r"(b.v[5]), "r"(b.v[6]), "r"(b.v[7]));
    reduce_once(s);  // a + b < 2p < 2^255: no carry out of limb 7
    return s;
}

__device__ __forceinline__ fe sub(const fe& a, const fe& b) {
    fe d;
    uint32_t br;
    asm("sub.cc.u32  %0, %9,  %17;\n\t"
        "subc.cc.u32 %1, %10, %18;\n\t"
        "subc.cc.u32 %2, %11, %19;\n\t"
        "subc.cc.u32 %3, %12, %20;\n\t"
        "subc.cc.u32 %4, %13, %21;\n\t"
        "subc.cc.u32 %5, %14, %22;\n\t"
        "subc.cc.u32 %6, %15, %23;\n\t"
        "subc.cc.u32 %7, %16, %24;\n\t"
        "subc.u32    %8, 0, 0;"
        : "=r"(d.v[0]), "=r"(d.v[1]), "=r"(d.v[2]), "=r"(d.v[3]), "=r"(d.v[4]), "=r"(d.v[5]), "=r"(d.v[6]), "=r"(d.v[7]), "=r"(br)
        : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]),
          "r"(b.v[0]), "r"(b.v[1]), "r"(b.v[2]), "r"(b.v[3]), "r"(b.v[4]), "r"(b.v[5]), "r"(b.v[6]), "r"(b.v[7]));
    // on borrow (br = 0xffffffff) add p back
    asm("add.cc.u32  %0, %0, %8;\n\t"
        "addc.cc.u32 %1, %1, %9;\n\t"
        "addc.cc.u32 %2, %2, %10;\n\t"
        "addc.cc.u32 %3, %3, %11;\n\t"
        "addc.cc.u32 %4, %4, %12;\n\t"
        "addc.cc.u32 %5, %5, %13;\n\t"
        "addc.cc.u32 %6, %6, %14;\n\t"
        "addc.u32    %7, %7, %15;"
        : "+r"(d.v[0]), "+r"(d.v[1]), "+r"(d.v[2]), "+r"(d.v[3]), "+r"(d.v[4]), "+r"(d.v[5]), "+r"(d.v[6]), "+r"(d.v[7])
        : "r"(FQ_P0 & br), "r"(FQ_P1 & br), "r"(FQ_P2 & br), "r"(FQ_P3 & br),
          "r"(FQ_P4 & br), "r"(FQ_P5 & br), "r"(FQ_P6 & br), "r"(FQ_P7 & br));
    return d;
}

__device__ __forceinline__ fe neg(const fe& a) {
    return is_zero(a) ? a : sub(zero(), a);
}

__device__ __forceinline__ fe dbl(const fe& a) { return add(a, a); }

// One CIOS round: t := (t + ai*b + m*p) / 2^32 with m chosen so the low limb
// cancels.  t holds 8 limbs on entry (limb 8 is implicitly zero).
__device__ __forceinline__ void cios_round(uint32_t& t0, uint32_t& t1, uint32_t& t2, uint32_t& t3,
                                           uint32_t& t4, uint32_t& t5, uint32_t& t6, uint32_t& t7,
                                           uint32_t ai, const fe& b) {
    asm("{\n\t"
        ".reg .u32 t8, m;\n\t"
        // t += lo(ai*b_j) at limb j
        "mad.lo.cc.u32  %0, %8, %9,  %0;\n\t"
        "madc.lo.cc.u32 %1, %8, %10, %1;\n\t"
        "madc.lo.cc.u32 %2, %8, %11, %2;\n\t"
        "madc.lo.cc.u32 %3, %8, %12, %3;\n\t"
        "madc.lo.cc.u32 %4, %8, %13, %4;\n\t"
        "madc.lo.cc.u32 %5, %8, %14, %5;\n\t"
        "madc.lo.cc.u32 %6, %8, %15, %6;\n\t"
        "madc.lo.cc.u32 %7, %8, %16, %7;\n\t"
        "addc.u32       t8, 0, 0;\n\t"
        // t += hi(ai*b_j) at limb j+1
        "mad.hi.cc.u32  %1, %8, %9,  %1;\n\t"
        "madc.hi.cc.u32 %2, %8, %10, %2;\n\t"
        "madc.hi.cc.u32 %3, %8, %11, %3;\n\t"
        "madc.hi.cc.u32 %4, %8, %12, %4;\n\t"
        "madc.hi.cc.u32 %5, %8, %13, %5;\n\t"
        "madc.hi.cc.u32 %6, %8, %14, %6;\n\t"
        "madc.hi.cc.u32 %7, %8, %15, %7;\n\t"
        "madc.hi.u32    t8, %8, %16, t8;\n\t"
        // m = t0 * (-p^-1) mod 2^32
        "mul.lo.u32     m, %0, %17;\n\t"
        // t += lo(m*p_j) at limb j (limb 0 becomes zero)
        "mad.lo.cc.u32  %0, m, %18, %0;\n\t"
        "madc.lo.cc.u32 %1, m, %19, %1;\n\t"
        "madc.lo.cc.u32 %2, m, %20, %2;\n\t"
        "madc.lo.cc.u32 %3, m, %21, %3;\n\t"
        "madc.lo.cc.u32 %4, m, %22, %4;\n\t"
        "madc.lo.cc.u32 %5, m, %23, %5;\n\t"
        "madc.lo.cc.u32 %6, m, %24, %6;\n\t"
        "madc.lo.cc.u32 %7, m, %25, %7;\n\t"
        "addc.u32       t8, t8, 0;\n\t"
        // t += hi(m*p_j) at limb j+1, written one limb down (the division by 2^32)
        "mad.hi.cc.u32  %0, m, %18, %1;\n\t"
        "madc.hi.cc.u32 %1, m, %19, %2;\n\t"
        "madc.hi.cc.u32 %2, m, %20, %3;\n\t"
        "madc.hi.cc.u32 %3, m, %21, %4;\n\t"
        "madc.hi.cc.u32 %4, m, %22, %5;\n\t"
        "madc.hi.cc.u32 %5, m, %23, %6;\n\t"
        "madc.hi.cc.u32 %6, m, %24, %7;\n\t"
        "madc.hi.u32    %7, m, %25, t8;\n\t"
        "}"
        : "+r"(t0), "+r"(t1), "+r"(t2), "+r"(t3), "+r"(t4), "+r"(t5), "+r"(t6), "+r"(t7)
        : "r"(ai), "r"(b.v[0]), "r"(b.v[1]), "r"(b.v[2]), "r"(b.v[3]), "r"(b.v[4]), "r"(b.v[5]), "r"(b.v[6]), "r"(b.v[7]),
          "n"(FQ_NP0), "n"(FQ_P0), "n"(FQ_P1), "n"(FQ_P2), "n"(FQ_P3), "n"(FQ_P4), "n"(FQ_P5), "n"(FQ_P6), "n"(FQ_P7));
}

// a * b * R^-1 mod p
__device__ __forceinline__ fe mul(const fe& a, const fe& b) {
    uint32_t t0 = 0, t1 = 0, t2 = 0, t3 = 0, t4 = 0, t5 = 0, t6 = 0, t7 = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) cios_round(t0, t1, t2, t3, t4, t5, t6, t7, a.v[i], b);
    fe r;
    r.v[0] = t0; r.v[1] = t1; r.v[2] = t2; r.v[3] = t3;
    r.v[4] = t4; r.v[5] = t5; r.v[6] = t6; r.v[7] = t7;
    reduce_once(r);
    return r;
}

__device__ __forceinline__ fe sqr(const fe& a) { return mul(a, a); }

__device__ __forceinline__ fe sqr_n(fe a, int n) {
    for (int i = 0; i < n; i++) a = sqr(a);
    return a;
}

// a^(p-2) = a^-1 (Fermat; p prime), inv(0) = 0.  Fixed 4-bit windows over the
// exponent p - 2, most significant first: 252 squarings and at most 63
// multiplications by the table entry a^w.
static __device__ __noinline__ fe inv_fermat(const fe& a) {
    // p - 2 in 4-bit digits, most significant first
    const uint32_t e[8] = {FQ_P7, FQ_P6, FQ_P5, FQ_P4, FQ_P3, FQ_P2, FQ_P1, FQ_P0 - 2u};
    fe tbl[16];
    tbl[0] = one();
    tbl[1] = a;
#pragma unroll 1
    for (int i = 2; i < 16; i++) tbl[i] = mul(tbl[i - 1], a);
    fe acc = one();
    bool started = false;
#pragma unroll 1
    for (int w = 0; w < 8; w++) {
#pragma unroll 1
        for (int nib = 7; nib >= 0; nib--) {
            uint32_t d = (e[w] >> (4 * nib)) & 0xF;
            if (started) acc = sqr_n(acc, 4);
            if (d) {
                acc = started ? mul(acc, tbl[d]) : tbl[d];
                started = true;
            }
        }
    }
    return acc;
}

// load / store helpers (16-byte vector access; caller guarantees alignment)
__device__ __forceinline__ fe load(const uint32_t* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    uint4 lo = q[0], hi = q[1];
    fe r;
    r.v[0] = lo.x; r.v[1] = lo.y; r.v[2] = lo.z; r.v[3] = lo.w;
    r.v[4] = hi.x; r.v[5] = hi.y; r.v[6] = hi.z; r.v[7] = hi.w;
    return r;
}

__device__ __forceinline__ void store(uint32_t* p, const fe& a) {
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = make_uint4(a.v[0], a.v[1], a.v[2], a.v[3]);
    q[1] = make_uint4(a.v[4], a.v[5], a.v[6], a.v[7]);
}

}  // namespace fq
