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
// Multiplication is Montgomery's REDC on the full product (separated operand
// scanning, see mul below).  Every carry chain sits in a single asm statement
// so that nothing can clobber the carry flag inside it.  On this part a lone
// 32-bit multiply-add issues in one slot of the multiply pipe for the low half
// and two for the high half, but a lo/hi pair over the same operands in one
// carry chain issues as one 64-bit multiply-add in two slots.  Every one of
// the 128 limb products of a multiplication is such a pair and the 8 reduction
// factors m are low-only, so a multiplication needs 264 slots: the roofline
// the kernels are measured against.
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

// Montgomery forms of 2, 3, 8 and 12 (k R mod p), so that a product by one of
// them is the plain multiple
#define FQ_MONT2 0x8b1e1b3au, 0xa6ba871bu, 0xeb8e167bu, 0x14f1d651u, 0xf0f28c58u, 0xccdd46deu, 0x340fbe5eu, 0x1c14ef83u
#define FQ_MONT3 0x50ad28d7u, 0x7a17caa9u, 0xe15521b9u, 0x1f6ac17au, 0x696bd284u, 0x334bea4eu, 0xce179d8eu, 0x2a1f6744u
#define FQ_MONT8 0x7b7e725au, 0x22a90440u, 0xdd54c4d4u, 0x24c48424u, 0xc0c780a5u, 0xc2d4900eu, 0x0ddbb927u, 0x0f8b2127u
#define FQ_MONT12 0xb93dab87u, 0x33fd8660u, 0x4bff273eu, 0xb726c637u, 0x212b40f7u, 0xa43ed816u, 0x94c995bbu, 0x1750b1bau

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

// Multiply-accumulate of one row, T[0..8] += x * (y_0 .. y_7), with the carry
// out of T[8] returned in cin (which holds, on entry, a carry to add into
// T[8]).  Each partial product is a lo/hi pair over the same operands written
// to adjacent limbs inside one carry chain (mad.lo.cc then madc.hi.cc): the
// compiler issues such a pair as a single 64-bit multiply-add, two issue
// slots of the multiply pipe instead of three for an unpaired lo and hi.  The
// even products y_0, y_2, y_4, y_6 fill limbs (0,1), (2,3), (4,5), (6,7) in
// one chain, the odd ones limbs (1,2) .. (7,8) in a second.
#define FQ_ROW_ASM                                \
    "{\n\t.reg .u32 c1;\n\t"                      \
    "mad.lo.cc.u32  %0, %10, %11, %0;\n\t"        \
    "madc.hi.cc.u32 %1, %10, %11, %1;\n\t"        \
    "madc.lo.cc.u32 %2, %10, %13, %2;\n\t"        \
    "madc.hi.cc.u32 %3, %10, %13, %3;\n\t"        \
    "madc.lo.cc.u32 %4, %10, %15, %4;\n\t"        \
    "madc.hi.cc.u32 %5, %10, %15, %5;\n\t"        \
    "madc.lo.cc.u32 %6, %10, %17, %6;\n\t"        \
    "madc.hi.cc.u32 %7, %10, %17, %7;\n\t"        \
    "addc.cc.u32    %8, %8, %9;\n\t"              \
    "addc.u32       c1, 0, 0;\n\t"                \
    "mad.lo.cc.u32  %1, %10, %12, %1;\n\t"        \
    "madc.hi.cc.u32 %2, %10, %12, %2;\n\t"        \
    "madc.lo.cc.u32 %3, %10, %14, %3;\n\t"        \
    "madc.hi.cc.u32 %4, %10, %14, %4;\n\t"        \
    "madc.lo.cc.u32 %5, %10, %16, %5;\n\t"        \
    "madc.hi.cc.u32 %6, %10, %16, %6;\n\t"        \
    "madc.lo.cc.u32 %7, %10, %18, %7;\n\t"        \
    "madc.hi.cc.u32 %8, %10, %18, %8;\n\t"        \
    "addc.u32       %9, c1, 0;\n\t"               \
    "}"
#define FQ_ROW_OUT(T, cin) \
    "+r"((T)[0]), "+r"((T)[1]), "+r"((T)[2]), "+r"((T)[3]), "+r"((T)[4]), "+r"((T)[5]), "+r"((T)[6]), "+r"((T)[7]), \
        "+r"((T)[8]), "+r"(cin)

__device__ __forceinline__ void mac_row(uint32_t* T, uint32_t& cin, uint32_t x, const uint32_t (&y)[8]) {
    asm(FQ_ROW_ASM
        : FQ_ROW_OUT(T, cin)
        : "r"(x), "r"(y[0]), "r"(y[1]), "r"(y[2]), "r"(y[3]), "r"(y[4]), "r"(y[5]), "r"(y[6]), "r"(y[7]));
}

// the same row with y = p (immediate operands)
__device__ __forceinline__ void mac_row_p(uint32_t* T, uint32_t& cin, uint32_t m) {
    asm(FQ_ROW_ASM
        : FQ_ROW_OUT(T, cin)
        : "r"(m), "n"(FQ_P0), "n"(FQ_P1), "n"(FQ_P2), "n"(FQ_P3), "n"(FQ_P4), "n"(FQ_P5), "n"(FQ_P6), "n"(FQ_P7));
}

// a * b * R^-1 mod p by separated operand scanning: the 512-bit product
// T = a b row by row (row i adds a_i b at limb i; its carry out of limb i+8
// starts limb i+9), then eight Montgomery rounds T += m p 2^(32 i) with
// m = T_i (-p^-1) mod 2^32, each of which zeroes limb i.  A round's carry out
// of limb i+8 belongs to limb i+9 and enters the next round's chain there.
// T stays below p^2 + p R < 2^511, so limb 16 and the last carry are zero, and
// T / R < 2p needs one conditional subtraction.
// The same without the final conditional subtraction: the result lies in
// [0, 2p) and is congruent to a b R^-1.  Valid whenever a b < p R, e.g. for
// a, b < 2p (4 p < R = 2^256), so such values may feed further lazy products.
__device__ __forceinline__ fe mul_lazy_inline(const fe& a, const fe& b) {
    uint32_t T[17];
#pragma unroll
    for (int i = 0; i < 17; i++) T[i] = 0;
    uint32_t cin;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        cin = 0;
        mac_row(T + i, cin, a.v[i], b.v);
        T[i + 9] = cin;
    }
    cin = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) mac_row_p(T + i, cin, T[i] * FQ_NP0);
    fe r;
#pragma unroll
    for (int j = 0; j < 8; j++) r.v[j] = T[8 + j];
    return r;
}

__device__ __forceinline__ fe mul_inline(const fe& a, const fe& b) {
    fe r = mul_lazy_inline(a, b);
    reduce_once(r);
    return r;
}

// a^2 * R^-1 mod p.  The 512-bit square is 2 (sum over i < j of a_i a_j
// 2^(32 (i + j))) + sum a_i^2 2^(64 i): seven triangular rows of the 28
// off-diagonal products (row i: a_i a_j for j > i, at limb 2i + 1 on, in two
// fused-pair chains like mac_row -- the even and the odd j -- each rippling its
// carry to the row's top limb i + 9, which no earlier row has reached), one
// doubling carry chain, and one chain of the 8 diagonal products as fused pairs
// at limbs (2i, 2i + 1).  36 limb products instead of 64: 208 issue slots of the
// multiply pipe instead of 264.  The Montgomery rounds are those of mul_inline.
__device__ __forceinline__ fe sqr_inline(const fe& a) {
    uint32_t T[17];
#pragma unroll
    for (int i = 0; i < 17; i++) T[i] = 0;
    asm("mad.lo.cc.u32 %0, %9, %10, %0;\n\t"
        "madc.hi.cc.u32 %1, %9, %10, %1;\n\t"
        "madc.lo.cc.u32 %2, %9, %12, %2;\n\t"
        "madc.hi.cc.u32 %3, %9, %12, %3;\n\t"
        "madc.lo.cc.u32 %4, %9, %14, %4;\n\t"
        "madc.hi.cc.u32 %5, %9, %14, %5;\n\t"
        "madc.lo.cc.u32 %6, %9, %16, %6;\n\t"
        "madc.hi.cc.u32 %7, %9, %16, %7;\n\t"
        "addc.u32 %8, %8, 0;\n\t"
        "mad.lo.cc.u32 %1, %9, %11, %1;\n\t"
        "madc.hi.cc.u32 %2, %9, %11, %2;\n\t"
        "madc.lo.cc.u32 %3, %9, %13, %3;\n\t"
        "madc.hi.cc.u32 %4, %9, %13, %4;\n\t"
        "madc.lo.cc.u32 %5, %9, %15, %5;\n\t"
        "madc.hi.cc.u32 %6, %9, %15, %6;\n\t"
        "addc.cc.u32 %7, %7, 0;\n\t"
        "addc.u32 %8, %8, 0;\n\t"
        : "+r"(T[1]), "+r"(T[2]), "+r"(T[3]), "+r"(T[4]), "+r"(T[5]), "+r"(T[6]), "+r"(T[7]), "+r"(T[8]), "+r"(T[9])
        : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %8, %9, %0;\n\t"
        "madc.hi.cc.u32 %1, %8, %9, %1;\n\t"
        "madc.lo.cc.u32 %2, %8, %11, %2;\n\t"
        "madc.hi.cc.u32 %3, %8, %11, %3;\n\t"
        "madc.lo.cc.u32 %4, %8, %13, %4;\n\t"
        "madc.hi.cc.u32 %5, %8, %13, %5;\n\t"
        "addc.cc.u32 %6, %6, 0;\n\t"
        "addc.u32 %7, %7, 0;\n\t"
        "mad.lo.cc.u32 %1, %8, %10, %1;\n\t"
        "madc.hi.cc.u32 %2, %8, %10, %2;\n\t"
        "madc.lo.cc.u32 %3, %8, %12, %3;\n\t"
        "madc.hi.cc.u32 %4, %8, %12, %4;\n\t"
        "madc.lo.cc.u32 %5, %8, %14, %5;\n\t"
        "madc.hi.cc.u32 %6, %8, %14, %6;\n\t"
        "addc.u32 %7, %7, 0;\n\t"
        : "+r"(T[3]), "+r"(T[4]), "+r"(T[5]), "+r"(T[6]), "+r"(T[7]), "+r"(T[8]), "+r"(T[9]), "+r"(T[10])
        : "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %7, %8, %0;\n\t"
        "madc.hi.cc.u32 %1, %7, %8, %1;\n\t"
        "madc.lo.cc.u32 %2, %7, %10, %2;\n\t"
        "madc.hi.cc.u32 %3, %7, %10, %3;\n\t"
        "madc.lo.cc.u32 %4, %7, %12, %4;\n\t"
        "madc.hi.cc.u32 %5, %7, %12, %5;\n\t"
        "addc.u32 %6, %6, 0;\n\t"
        "mad.lo.cc.u32 %1, %7, %9, %1;\n\t"
        "madc.hi.cc.u32 %2, %7, %9, %2;\n\t"
        "madc.lo.cc.u32 %3, %7, %11, %3;\n\t"
        "madc.hi.cc.u32 %4, %7, %11, %4;\n\t"
        "addc.cc.u32 %5, %5, 0;\n\t"
        "addc.u32 %6, %6, 0;\n\t"
        : "+r"(T[5]), "+r"(T[6]), "+r"(T[7]), "+r"(T[8]), "+r"(T[9]), "+r"(T[10]), "+r"(T[11])
        : "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %6, %7, %0;\n\t"
        "madc.hi.cc.u32 %1, %6, %7, %1;\n\t"
        "madc.lo.cc.u32 %2, %6, %9, %2;\n\t"
        "madc.hi.cc.u32 %3, %6, %9, %3;\n\t"
        "addc.cc.u32 %4, %4, 0;\n\t"
        "addc.u32 %5, %5, 0;\n\t"
        "mad.lo.cc.u32 %1, %6, %8, %1;\n\t"
        "madc.hi.cc.u32 %2, %6, %8, %2;\n\t"
        "madc.lo.cc.u32 %3, %6, %10, %3;\n\t"
        "madc.hi.cc.u32 %4, %6, %10, %4;\n\t"
        "addc.u32 %5, %5, 0;\n\t"
        : "+r"(T[7]), "+r"(T[8]), "+r"(T[9]), "+r"(T[10]), "+r"(T[11]), "+r"(T[12])
        : "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %5, %6, %0;\n\t"
        "madc.hi.cc.u32 %1, %5, %6, %1;\n\t"
        "madc.lo.cc.u32 %2, %5, %8, %2;\n\t"
        "madc.hi.cc.u32 %3, %5, %8, %3;\n\t"
        "addc.u32 %4, %4, 0;\n\t"
        "mad.lo.cc.u32 %1, %5, %7, %1;\n\t"
        "madc.hi.cc.u32 %2, %5, %7, %2;\n\t"
        "addc.cc.u32 %3, %3, 0;\n\t"
        "addc.u32 %4, %4, 0;\n\t"
        : "+r"(T[9]), "+r"(T[10]), "+r"(T[11]), "+r"(T[12]), "+r"(T[13])
        : "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %4, %5, %0;\n\t"
        "madc.hi.cc.u32 %1, %4, %5, %1;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.u32 %3, %3, 0;\n\t"
        "mad.lo.cc.u32 %1, %4, %6, %1;\n\t"
        "madc.hi.cc.u32 %2, %4, %6, %2;\n\t"
        "addc.u32 %3, %3, 0;\n\t"
        : "+r"(T[11]), "+r"(T[12]), "+r"(T[13]), "+r"(T[14])
        : "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\t"
        "madc.hi.cc.u32 %1, %3, %4, %1;\n\t"
        "addc.u32 %2, %2, 0;\n\t"
        : "+r"(T[13]), "+r"(T[14]), "+r"(T[15])
        : "r"(a.v[6]), "r"(a.v[7]));
    // T = 2 T (the off-diagonal sum is below 2^510)
    asm("add.cc.u32  %0, %0, %0;\n\t"
        "addc.cc.u32 %1, %1, %1;\n\t"
        "addc.cc.u32 %2, %2, %2;\n\t"
        "addc.cc.u32 %3, %3, %3;\n\t"
        "addc.cc.u32 %4, %4, %4;\n\t"
        "addc.cc.u32 %5, %5, %5;\n\t"
        "addc.cc.u32 %6, %6, %6;\n\t"
        "addc.cc.u32 %7, %7, %7;\n\t"
        "addc.cc.u32 %8, %8, %8;\n\t"
        "addc.cc.u32 %9, %9, %9;\n\t"
        "addc.cc.u32 %10, %10, %10;\n\t"
        "addc.cc.u32 %11, %11, %11;\n\t"
        "addc.cc.u32 %12, %12, %12;\n\t"
        "addc.cc.u32 %13, %13, %13;\n\t"
        "addc.cc.u32 %14, %14, %14;\n\t"
        "addc.u32    %15, %15, %15;"
        : "+r"(T[0]), "+r"(T[1]), "+r"(T[2]), "+r"(T[3]), "+r"(T[4]), "+r"(T[5]), "+r"(T[6]), "+r"(T[7]), "+r"(T[8]), "+r"(T[9]), "+r"(T[10]), "+r"(T[11]), "+r"(T[12]), "+r"(T[13]), "+r"(T[14]), "+r"(T[15]));
    // T += sum_i a_i^2 2^(64 i); the square is below 2^512, no carry out
    asm("mad.lo.cc.u32  %0, %16, %16, %0;\n\t"
        "madc.hi.cc.u32 %1, %16, %16, %1;\n\t"
        "madc.lo.cc.u32 %2, %17, %17, %2;\n\t"
        "madc.hi.cc.u32 %3, %17, %17, %3;\n\t"
        "madc.lo.cc.u32 %4, %18, %18, %4;\n\t"
        "madc.hi.cc.u32 %5, %18, %18, %5;\n\t"
        "madc.lo.cc.u32 %6, %19, %19, %6;\n\t"
        "madc.hi.cc.u32 %7, %19, %19, %7;\n\t"
        "madc.lo.cc.u32 %8, %20, %20, %8;\n\t"
        "madc.hi.cc.u32 %9, %20, %20, %9;\n\t"
        "madc.lo.cc.u32 %10, %21, %21, %10;\n\t"
        "madc.hi.cc.u32 %11, %21, %21, %11;\n\t"
        "madc.lo.cc.u32 %12, %22, %22, %12;\n\t"
        "madc.hi.cc.u32 %13, %22, %22, %13;\n\t"
        "madc.lo.cc.u32 %14, %23, %23, %14;\n\t"
        "madc.hi.u32    %15, %23, %23, %15;"
        : "+r"(T[0]), "+r"(T[1]), "+r"(T[2]), "+r"(T[3]), "+r"(T[4]), "+r"(T[5]), "+r"(T[6]), "+r"(T[7]), "+r"(T[8]), "+r"(T[9]), "+r"(T[10]), "+r"(T[11]), "+r"(T[12]), "+r"(T[13]), "+r"(T[14]), "+r"(T[15])
        : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]), "r"(a.v[6]), "r"(a.v[7]));
    uint32_t cin = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) mac_row_p(T + i, cin, T[i] * FQ_NP0);
    fe r;
#pragma unroll
    for (int j = 0; j < 8; j++) r.v[j] = T[8 + j];
    reduce_once(r);
    return r;
}

// Called, not inlined: every kernel of the MSM runs long sequences of field
// multiplications, and inlining each ~330-instruction body at every call site
// makes the hot loops overflow the per-sub-partition instruction cache (the
// warps then stall waiting for instruction fetch).  One shared body stays
// resident.  The operands are taken by value: a reference parameter of a called function
// makes the caller store the operand to its stack frame and the callee load it
// back, two round trips through local memory per multiplication.
static __device__ __noinline__ fe mul(fe a, fe b) { return mul_inline(a, b); }
static __device__ __noinline__ fe mul_lazy(fe a, fe b) { return mul_lazy_inline(a, b); }

// sqr_fused (called, like mul) issues fewer multiply-pipe slots but its three
// chains (rows, doubling, diagonal) are more serial than a multiplication's
// rows: it pays in the throughput-bound batched additions (n = 2^22: tree
// levels 5.72 -> 5.58 ms) and costs in the latency-bound Jacobian chains of the
// bucket reduction (0.49 -> 0.53 ms), which therefore square by multiplying.
static __device__ __noinline__ fe sqr_fused(fe a) { return sqr_inline(a); }

__device__ __forceinline__ fe sqr(const fe& a) { return mul(a, a); }

__device__ __forceinline__ fe sqr_n(fe a, int n) {
    for (int i = 0; i < n; i++) a = sqr(a);
    return a;
}

// a^(p-2) = a^-1 (Fermat; p prime), inv(0) = 0.  Fixed 4-bit windows over the
// exponent p - 2, most significant first: 252 squarings and at most 63
// multiplications by the table entry a^w.
static __device__ __noinline__ fe inv_fermat(fe a) {
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
