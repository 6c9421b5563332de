// msm_testing.cu -- test hooks: single device primitives of the MSM path run
// over arrays, so that each can be compared with the CPU oracle.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/msm_g1_testing.h"
#include "g1_coop.cuh"
#include "g1_proj.cuh"
#include "msm_core.cuh"

using fq::fe;
using g1::aff;
using g1::jac;

namespace {

__global__ void k_test_fq(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n) {
    __shared__ uint32_t divtab[inv::kDivTabEntries];
    inv::load_divtab(divtab);
    __syncthreads();
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (op == MSM_G1_TEST_FQ_INV_BLOCK) {  // the whole block takes part; past the end it inverts one
        __shared__ uint32_t sh[8 * 128];
        const fe r = msm::block_inverse(i < n ? fq::load(a + 8 * i) : fq::one(), sh, 0, divtab);
        if (i < n) fq::store(out + 8 * i, r);
        return;
    }
    if (i >= n) return;
    fe x = fq::load(a + 8 * i);
    fe r;
    switch (op) {
        case MSM_G1_TEST_FQ_MUL: r = fq::mul(x, fq::load(b + 8 * i)); break;
        case MSM_G1_TEST_FQ_SQR: r = fq::sqr_fused(x); break;  // the fused-pair squaring
        case MSM_G1_TEST_FQ_ADD: r = fq::add(x, fq::load(b + 8 * i)); break;
        case MSM_G1_TEST_FQ_SUB: r = fq::sub(x, fq::load(b + 8 * i)); break;
        case MSM_G1_TEST_FQ_NEG: r = fq::neg(x); break;
        case MSM_G1_TEST_FQ_INV: r = inv::inv_safegcd(x); break;
        case MSM_G1_TEST_FQ_INV_TABLE: r = inv::inv_safegcd_tab(x, divtab); break;
        default: r = fq::inv_fermat(x); break;
    }
    fq::store(out + 8 * i, r);
}

__global__ void k_test_g1(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    switch (op) {
        case MSM_G1_TEST_JAC_DBL: g1::store_jac(out + 24 * i, g1::dbl(g1::load_jac(a + 24 * i))); break;
        case MSM_G1_TEST_JAC_ADD:
            g1::store_jac(out + 24 * i, g1::add(g1::load_jac(a + 24 * i), g1::load_jac(b + 24 * i)));
            break;
        case MSM_G1_TEST_JAC_MIXED:
            g1::store_jac(out + 24 * i, g1::add_mixed(g1::load_jac(a + 24 * i), g1::load_aff(b + 16 * i)));
            break;
        case MSM_G1_TEST_AFF_ADD:
            g1::store_jac(out + 24 * i, g1::add_aff(g1::load_aff(a + 16 * i), g1::load_aff(b + 16 * i)));
            break;
        default: g1::store_aff(out + 16 * i, g1::to_aff(g1::load_jac(a + 24 * i))); break;
    }
}

// one group of W lanes per element (W = 32: a warp; W = 8: four elements per
// warp, whose groups may take different branches), all lanes of a group
// holding the same operands
template <int W>
__global__ void k_test_g1_coop(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n) {
    size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / W;
    if (i >= n) return;
    jac r;
    if (op == MSM_G1_TEST_JAC_DBL_COOP || op == MSM_G1_TEST_JAC_DBL_COOP8)
        r = g1c::dbl<W>(g1::load_jac(a + 24 * i));
    else if (op == MSM_G1_TEST_JAC_DBL5_COOP)
        r = g1c::dbl_n<W>(g1::load_jac(a + 24 * i), 5);
    else if (op == MSM_G1_TEST_JAC_ADD_COOP || op == MSM_G1_TEST_JAC_ADD_COOP8)
        r = g1c::add<W>(g1::load_jac(a + 24 * i), g1::load_jac(b + 24 * i));
    else
        r = g1c::add_mixed<W>(g1::load_jac(a + 24 * i), g1::load_aff(b + 16 * i));
    if ((threadIdx.x & (W - 1)) == 0) g1::store_jac(out + 24 * i, r);
}

// The residue-number-system chains, one warp per element.
__global__ void __launch_bounds__(64) k_test_rns(int op, const uint32_t* a, const uint32_t* b, uint32_t* out,
                                                 size_t n, int arg) {
    __shared__ __align__(16) uint32_t xch[g1p::kXchWords];
    const size_t i = blockIdx.x;
    if (i >= n) return;
    const bool t0 = threadIdx.x == 0;
    if (op == MSM_G1_TEST_RNS_DBL_N || op == MSM_G1_TEST_RNS_ADD || op == MSM_G1_TEST_RNS_HORNER) {
        // the two-warp chains of g1_proj.cuh
        g1p::Pair P = g1p::make_pair(xch);
        jac o;
        if (op == MSM_G1_TEST_RNS_DBL_N) {
            o = g1p::dbl_n_positional(P, g1::load_jac(a + 24 * i), arg);
        } else if (op == MSM_G1_TEST_RNS_ADD) {
            const g1p::rproj pa = g1p::to_proj(P, g1::load_jac(a + 24 * i));
            const g1p::rproj pb = g1p::to_proj(P, g1::load_jac(b + 24 * i));
            o = g1p::to_jac(P, g1p::add(P, pa, pb));
        } else {
            // a holds arg window sums (24 words each) for element i, top window last; width 13 each
            const uint32_t* ws = a + (size_t)24 * arg * i;
            o = g1p::horner(P, g1::load_jac(ws + 24 * (arg - 1)), arg - 2, 0, [](int) { return 13; },
                            [&](int w) { return g1::load_jac(ws + 24 * w); });
        }
        if (t0) g1::store_jac(out + 24 * i, o);
        return;
    }
    if (threadIdx.x >= 32) return;  // one warp
    const rns::Ctx C = rns::make_ctx();
    switch (op) {
        case MSM_G1_TEST_RNS_MUL:
        case MSM_G1_TEST_RNS_SQR_CHAIN: {
            const rns::rv x = rns::mm(C, rns::residues(C, fq::load(a + 8 * i)), rns::cin(C));
            rns::rv r;
            if (op == MSM_G1_TEST_RNS_MUL) {
                r = rns::mm(C, x, rns::mm(C, rns::residues(C, fq::load(b + 8 * i)), rns::cin(C)));
            } else {  // x^(2^arg), each square from the previous lazily reduced value
                r = x;
                for (int k = 0; k < arg; k++) r = rns::mm(C, r, r);
            }
            const fq::fe o = rns::to_positional(C, rns::mm(C, r, rns::cout(C)));
            if (t0) fq::store(out + 8 * i, o);
            break;
        }
        default: {  // MSM_G1_TEST_RNS_IS_ZERO: the integer a (8 words) below arg * p, as residues
            const bool z = rns::is_zero(C, rns::residues(C, fq::load(a + 8 * i)), (uint32_t)arg);
            if (t0) out[i] = z ? 1u : 0u;
            break;
        }
    }
}

template <int S>
struct PairArraySrc {
    const uint32_t *a, *b;
    uint32_t* out;
    size_t i0;
    __device__ __forceinline__ bool has_q(int) const { return true; }
    __device__ __forceinline__ fe xp(int k) const { return fq::load(a + 16 * (i0 + k)); }
    __device__ __forceinline__ fe xq(int k) const { return fq::load(b + 16 * (i0 + k)); }
    __device__ __forceinline__ void ys(int k, fe& ya, fe& yb) const {
        ya = fq::load(a + 16 * (i0 + k) + 8);
        yb = fq::load(b + 16 * (i0 + k) + 8);
    }
    __device__ __forceinline__ aff p(int k) const { return g1::load_aff(a + 16 * (i0 + k)); }
    __device__ __forceinline__ aff q(int k) const { return g1::load_aff(b + 16 * (i0 + k)); }
    __device__ __forceinline__ void store(int k, const aff& r) { g1::store_aff(out + 16 * (i0 + k), r); }
};

// block: the block's threads share one inversion (all of them call, those
// past the end with no pairs), as in the accumulation kernels
template <int S, bool INLINE_BACK>
__global__ void k_test_batch_add(const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n, int block) {
    __shared__ uint32_t sh[8 * 256];
    size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t i0 = t * S;
    if (block ? (size_t)blockIdx.x * blockDim.x * S >= n : i0 >= n) return;
    int count = i0 >= n ? 0 : (int)((n - i0) < (size_t)S ? (n - i0) : (size_t)S);
    PairArraySrc<S> src{a, b, out, i0};
    msm::batch_pairs<S, INLINE_BACK>(src, count, 0, block ? sh : nullptr);
}

__global__ void k_test_digits(const uint32_t* scalars, size_t n, int c, int nbits, int32_t* digits) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t k[8];
    msm::load_scalar(scalars + 8 * i, k);
    msm::reduce_mod_r(k);
    const msm::Windows L = msm::make_windows(c, nbits);
    uint32_t carry = 0;
    for (int w = 0; w < L.W; w++) digits[i * L.W + w] = msm::signed_digit(k, L, w, carry);
}

__global__ void k_test_glv_split(const uint32_t* scalars, size_t n, uint32_t* out) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t k[8], k1[4], k2[4], s1, s2;
    msm::load_scalar(scalars + 8 * i, k);
    msm::reduce_mod_r(k);
    glv::split(k, k1, k2, s1, s2);
    for (int j = 0; j < 4; j++) {
        out[i * 10 + j] = k1[j];
        out[i * 10 + 4 + j] = k2[j];
    }
    out[i * 10 + 8] = s1;
    out[i * 10 + 9] = s2;
}

bool a16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

extern "C" int msm_g1_test_fq(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n,
                              cudaStream_t st) {
    if (op < MSM_G1_TEST_FQ_MUL || op > MSM_G1_TEST_FQ_INV_BLOCK) return MSM_G1_ERR_INVALID_ARG;
    bool needs_b = op == MSM_G1_TEST_FQ_MUL || op == MSM_G1_TEST_FQ_ADD || op == MSM_G1_TEST_FQ_SUB;
    if (n == 0) return MSM_G1_OK;
    if (!a || !out || !a16(a) || !a16(out) || (needs_b && (!b || !a16(b)))) return MSM_G1_ERR_INVALID_ARG;
    k_test_fq<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(op, a, b, out, n);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_test_g1(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n,
                              cudaStream_t st) {
    if (op < MSM_G1_TEST_JAC_DBL || op > MSM_G1_TEST_AFF_ADD) return MSM_G1_ERR_INVALID_ARG;
    bool needs_b = op != MSM_G1_TEST_JAC_DBL && op != MSM_G1_TEST_TO_AFFINE && op != MSM_G1_TEST_JAC_DBL_COOP &&
                   op != MSM_G1_TEST_JAC_DBL_COOP8 && op != MSM_G1_TEST_JAC_DBL5_COOP;
    if (n == 0) return MSM_G1_OK;
    if (!a || !out || !a16(a) || !a16(out) || (needs_b && (!b || !a16(b)))) return MSM_G1_ERR_INVALID_ARG;
    if (op >= MSM_G1_TEST_JAC_DBL_COOP8 && op <= MSM_G1_TEST_JAC_MIXED_COOP8)
        k_test_g1_coop<8><<<(unsigned)((n * 8 + 127) / 128), 128, 0, st>>>(op, a, b, out, n);
    else if (op >= MSM_G1_TEST_JAC_DBL_COOP && op <= MSM_G1_TEST_JAC_DBL5_COOP)
        k_test_g1_coop<32><<<(unsigned)((n * 32 + 127) / 128), 128, 0, st>>>(op, a, b, out, n);
    else
        k_test_g1<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(op, a, b, out, n);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_test_rns(int op, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n, int arg,
                               cudaStream_t st) {
    if (op < MSM_G1_TEST_RNS_MUL || op > MSM_G1_TEST_RNS_IS_ZERO || arg < 0) return MSM_G1_ERR_INVALID_ARG;
    if (n == 0) return MSM_G1_OK;
    const bool needs_b = op == MSM_G1_TEST_RNS_MUL || op == MSM_G1_TEST_RNS_ADD;
    if (!a || !out || !a16(a) || (needs_b && (!b || !a16(b)))) return MSM_G1_ERR_INVALID_ARG;
    if (op == MSM_G1_TEST_RNS_HORNER && arg < 1) return MSM_G1_ERR_INVALID_ARG;
    k_test_rns<<<(unsigned)n, 64, 0, st>>>(op, a, b, out, n, arg);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_test_batch_add(const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n, int batch_s,
                                     int mode, cudaStream_t st) {
    if (n == 0) return MSM_G1_OK;
    if (!a || !b || !out || !a16(a) || !a16(b) || !a16(out) || mode < 0 || mode > 3) return MSM_G1_ERR_INVALID_ARG;
    const bool inline_back = mode & 1;
    const int block = (mode >> 1) & 1;
    size_t threads;
    switch (batch_s) {
#define CASE(S)                                                                                  \
    case S:                                                                                      \
        threads = (n + S - 1) / S;                                                               \
        if (inline_back)                                                                         \
            k_test_batch_add<S, true><<<(unsigned)((threads + 127) / 128), 128, 0, st>>>(a, b, out, n, block); \
        else                                                                                     \
            k_test_batch_add<S, false><<<(unsigned)((threads + 127) / 128), 128, 0, st>>>(a, b, out, n, block); \
        break;
        CASE(1) CASE(2) CASE(4) CASE(8) CASE(16) CASE(32) CASE(64)
#undef CASE
        default: return MSM_G1_ERR_INVALID_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_test_digits(const uint32_t* scalars, size_t n, int c, int nbits, int32_t* digits,
                                  cudaStream_t st) {
    if (c < 1 || c > MSM_G1_MAX_WINDOW) return MSM_G1_ERR_INVALID_ARG;
    if (nbits != msm::PLAIN_BITS && nbits != msm::GLV_BITS) return MSM_G1_ERR_INVALID_ARG;
    if (n == 0) return MSM_G1_OK;
    if (!scalars || !digits || !a16(scalars)) return MSM_G1_ERR_INVALID_ARG;
    k_test_digits<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(scalars, n, c, nbits, digits);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_test_glv_split(const uint32_t* scalars, size_t n, uint32_t* out, cudaStream_t st) {
    if (n == 0) return MSM_G1_OK;
    if (!scalars || !out || !a16(scalars)) return MSM_G1_ERR_INVALID_ARG;
    k_test_glv_split<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(scalars, n, out);
    return cudaGetLastError() == cudaSuccess ? MSM_G1_OK : MSM_G1_ERR_CUDA;
}

extern "C" int msm_g1_glv_constants(uint32_t* beta_mont, uint32_t* lambda) {
    if (!beta_mont || !lambda) return MSM_G1_ERR_INVALID_ARG;
    const uint32_t b[8] = {GLV_BETA_MONT}, l[8] = {GLV_LAMBDA};
    for (int j = 0; j < 8; j++) {
        beta_mont[j] = b[j];
        lambda[j] = l[j];
    }
    return MSM_G1_OK;
}
