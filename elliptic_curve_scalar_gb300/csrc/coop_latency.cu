// coop_latency.cu -- latency of the warp-cooperative point operations of the
// window combination and the bucket reduction (g1_coop.cuh), one warp, one
// chain of dependent operations.  Standalone program:
//   nvcc -O3 -std=c++17 -gencode arch=compute_103a,code=sm_103a \
//        -o coop_latency elliptic_curve_scalar_gb300/csrc/coop_latency.cu && ./coop_latency
// Prints cycles per operation (clock64 around 1024 dependent operations) for
// g1c::dbl applied repeatedly, the doubling chain g1c::dbl_n (constants folded
// into the products), g1c::add and one field multiplication, and checks that
// both doubling forms give the same Jacobian point.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "g1_coop.cuh"

using fq::fe;
using g1::jac;

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s @%d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

template <int V>
__global__ void k_chain(const uint32_t* in, uint32_t* out, int n, long long* cyc) {
    jac p = g1::load_jac(in), q = g1::load_jac(in + 24);
    fe a = p.X, b = q.X;
    __syncwarp();
    long long t0 = clock64();
    if (V == 0) {
        for (int i = 0; i < n; i++) p = g1c::dbl(p);
    } else if (V == 1) {
        p = g1c::dbl_n(p, n);
    } else if (V == 2) {
        for (int i = 0; i < n; i++) p = g1c::add(p, q);
    } else {
        for (int i = 0; i < n; i++) a = fq::mul_inline(a, b);
        p.X = a;
    }
    __syncwarp();
    long long t1 = clock64();
    if (threadIdx.x == 0) {
        g1::store_jac(out, p);
        cyc[0] = t1 - t0;
    }
}

int main() {
    // G = (1, 2) with Z = 1 in Montgomery form, and q = G + G from the library's own doubling
    const uint32_t one[8] = {FQ_R0, FQ_R1, FQ_R2, FQ_R3, FQ_R4, FQ_R5, FQ_R6, FQ_R7};
    const uint32_t two[8] = {FQ_MONT2};
    uint32_t h_in[48];
    for (int i = 0; i < 8; i++) {
        h_in[i] = one[i];
        h_in[8 + i] = two[i];
        h_in[16 + i] = one[i];
    }
    for (int i = 0; i < 24; i++) h_in[24 + i] = h_in[i];
    uint32_t *d_in, *d_out;
    long long* d_cyc;
    CK(cudaMalloc(&d_in, 192));
    CK(cudaMalloc(&d_out, 4 * 96));
    CK(cudaMalloc(&d_cyc, 4 * 8));
    CK(cudaMemcpy(d_in, h_in, 192, cudaMemcpyHostToDevice));
    k_chain<0><<<1, 32>>>(d_in, d_out, 1, d_cyc);  // q = 2G
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(h_in + 24, d_out, 96, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(d_in, h_in, 192, cudaMemcpyHostToDevice));
    const int n = 1024;
    k_chain<0><<<1, 32>>>(d_in, d_out + 0, n, d_cyc + 0);
    k_chain<1><<<1, 32>>>(d_in, d_out + 24, n, d_cyc + 1);
    k_chain<2><<<1, 32>>>(d_in, d_out + 48, n, d_cyc + 2);
    k_chain<3><<<1, 32>>>(d_in, d_out + 72, n, d_cyc + 3);
    CK(cudaDeviceSynchronize());
    long long cyc[4];
    uint32_t h_out[96];
    CK(cudaMemcpy(cyc, d_cyc, 32, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(h_out, d_out, 4 * 96, cudaMemcpyDeviceToHost));
    bool same = true;
    for (int i = 0; i < 24; i++) same = same && h_out[i] == h_out[24 + i];
    printf("g1c::dbl, repeated             %8.1f cycles per doubling\n", (double)cyc[0] / n);
    printf("g1c::dbl_n (constants folded)  %8.1f cycles per doubling\n", (double)cyc[1] / n);
    printf("g1c::add                       %8.1f cycles per addition\n", (double)cyc[2] / n);
    printf("fq::mul_inline, one warp       %8.1f cycles per multiplication\n", (double)cyc[3] / n);
    printf("dbl and dbl_n agree: %s\n", same ? "yes" : "NO");
    return same ? 0 : 1;
}
