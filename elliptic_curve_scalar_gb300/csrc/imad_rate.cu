// imad_rate.cu -- measures the 32-bit integer multiply pipe of this GPU and
// the library's field multiplication: the denominator of the IMAD roofline
// bench.py reports.  Standalone program:
//   nvcc -O3 -std=c++17 -gencode arch=compute_103a,code=sm_103a \
//        -o imad_rate elliptic_curve_scalar_gb300/csrc/imad_rate.cu && ./imad_rate
// Prints mad.lo / mad.hi / carry-chained madc throughput (ops/s), the rate of
// full limb products issued as lo/hi pairs in one carry chain (the form the
// field multiplication uses) and as unpaired lo and hi, dependent latencies
// (cycles), and the latency and throughput of fq::mul and fq::sqr_fused.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "fq.cuh"

using fq::fe;

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s @%d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

// ---------- raw IMAD throughput: 8 independent mad.lo chains per thread
__global__ void k_imad_tput(uint32_t* out, int iters, uint32_t seed) {
    uint32_t a0 = seed + threadIdx.x, a1 = a0 ^ 1, a2 = a0 ^ 2, a3 = a0 ^ 3, a4 = a0 ^ 4, a5 = a0 ^ 5, a6 = a0 ^ 6, a7 = a0 ^ 7;
    uint32_t b = seed * 3 + 1;
    for (int i = 0; i < iters; i++) {
        asm volatile("mad.lo.u32 %0, %0, %8, %0;\n\t"
                     "mad.lo.u32 %1, %1, %8, %1;\n\t"
                     "mad.lo.u32 %2, %2, %8, %2;\n\t"
                     "mad.lo.u32 %3, %3, %8, %3;\n\t"
                     "mad.lo.u32 %4, %4, %8, %4;\n\t"
                     "mad.lo.u32 %5, %5, %8, %5;\n\t"
                     "mad.lo.u32 %6, %6, %8, %6;\n\t"
                     "mad.lo.u32 %7, %7, %8, %7;"
                     : "+r"(a0), "+r"(a1), "+r"(a2), "+r"(a3), "+r"(a4), "+r"(a5), "+r"(a6), "+r"(a7) : "r"(b));
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = a0 ^ a1 ^ a2 ^ a3 ^ a4 ^ a5 ^ a6 ^ a7;
}

__global__ void k_imadhi_tput(uint32_t* out, int iters, uint32_t seed) {
    uint32_t a0 = seed + threadIdx.x, a1 = a0 ^ 1, a2 = a0 ^ 2, a3 = a0 ^ 3, a4 = a0 ^ 4, a5 = a0 ^ 5, a6 = a0 ^ 6, a7 = a0 ^ 7;
    uint32_t b = seed * 3 + 1;
    for (int i = 0; i < iters; i++) {
        asm volatile("mad.hi.u32 %0, %0, %8, %0;\n\t"
                     "mad.hi.u32 %1, %1, %8, %1;\n\t"
                     "mad.hi.u32 %2, %2, %8, %2;\n\t"
                     "mad.hi.u32 %3, %3, %8, %3;\n\t"
                     "mad.hi.u32 %4, %4, %8, %4;\n\t"
                     "mad.hi.u32 %5, %5, %8, %5;\n\t"
                     "mad.hi.u32 %6, %6, %8, %6;\n\t"
                     "mad.hi.u32 %7, %7, %8, %7;"
                     : "+r"(a0), "+r"(a1), "+r"(a2), "+r"(a3), "+r"(a4), "+r"(a5), "+r"(a6), "+r"(a7) : "r"(b));
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = a0 ^ a1 ^ a2 ^ a3 ^ a4 ^ a5 ^ a6 ^ a7;
}

// carry-chained madc (4 independent chains of length 8 per iteration, in separate asm blocks)
__global__ void k_madc_tput(uint32_t* out, int iters, uint32_t seed) {
    uint32_t t[4][8];
    for (int c = 0; c < 4; c++) for (int j = 0; j < 8; j++) t[c][j] = seed + c * 8 + j + threadIdx.x;
    uint32_t b = seed * 5 + 3;
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int c = 0; c < 4; c++)
            asm volatile("mad.lo.cc.u32  %0, %8, %0, %1;\n\t"
                         "madc.lo.cc.u32 %1, %8, %1, %2;\n\t"
                         "madc.lo.cc.u32 %2, %8, %2, %3;\n\t"
                         "madc.lo.cc.u32 %3, %8, %3, %4;\n\t"
                         "madc.lo.cc.u32 %4, %8, %4, %5;\n\t"
                         "madc.lo.cc.u32 %5, %8, %5, %6;\n\t"
                         "madc.lo.cc.u32 %6, %8, %6, %7;\n\t"
                         "madc.lo.u32    %7, %8, %7, %0;"
                         : "+r"(t[c][0]), "+r"(t[c][1]), "+r"(t[c][2]), "+r"(t[c][3]), "+r"(t[c][4]), "+r"(t[c][5]),
                           "+r"(t[c][6]), "+r"(t[c][7])
                         : "r"(b));
    }
    uint32_t x = 0;
    for (int c = 0; c < 4; c++) for (int j = 0; j < 8; j++) x ^= t[c][j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = x;
}

// ---------- full limb products: rows of lo/hi pairs over the same operands
// (fq::mac_row), two independent rows of 8 products per iteration
__global__ void k_pair_row_tput(uint32_t* out, int iters, uint32_t seed) {
    uint32_t t[2][9], cin[2] = {0, 0};
    for (int c = 0; c < 2; c++) for (int j = 0; j < 9; j++) t[c][j] = seed + c * 9 + j + threadIdx.x;
    uint32_t b[8];
    for (int j = 0; j < 8; j++) b[j] = seed * (j + 3) + 1;
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int c = 0; c < 2; c++) fq::mac_row(t[c], cin[c], (uint32_t)i * 0x9e3779b9u + (uint32_t)c, b);
    }
    uint32_t x = cin[0] ^ cin[1];
    for (int c = 0; c < 2; c++) for (int j = 0; j < 9; j++) x ^= t[c][j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = x;
}

// unpaired: 8 mad.hi and 8 mad.lo on different operands per iteration
__global__ void k_unpaired_tput(uint32_t* out, int iters, uint32_t seed) {
    uint32_t h[8], l[8];
    for (int j = 0; j < 8; j++) { h[j] = seed + threadIdx.x + j; l[j] = h[j] * 7; }
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int j = 0; j < 8; j++) {
            asm volatile("mad.hi.u32 %0, %0, %1, %0;" : "+r"(h[j]) : "r"(l[j]));
            asm volatile("mad.lo.u32 %0, %0, %1, %0;" : "+r"(l[j]) : "r"(h[j]));
        }
    }
    uint32_t x = 0;
    for (int j = 0; j < 8; j++) x ^= h[j] ^ l[j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = x;
}

// ---------- raw IMAD latency (single thread)
__global__ void k_imad_lat(uint32_t* out, int iters, uint32_t seed, long long* cyc) {
    uint32_t a = seed, b = seed * 3 + 1;
    long long t0 = clock64();
    for (int i = 0; i < iters; i++) {
        asm volatile("mad.lo.u32 %0, %0, %1, %0;\n\t"
                     "mad.lo.u32 %0, %0, %1, %0;\n\t"
                     "mad.lo.u32 %0, %0, %1, %0;\n\t"
                     "mad.lo.u32 %0, %0, %1, %0;" : "+r"(a) : "r"(b));
    }
    long long t1 = clock64();
    out[0] = a;
    cyc[0] = t1 - t0;
}

__global__ void k_madc_lat(uint32_t* out, int iters, uint32_t seed, long long* cyc) {
    uint32_t t0_ = seed, t1_ = seed + 1, t2_ = seed + 2, t3_ = seed + 3;
    uint32_t b = seed * 3 + 1;
    long long t0 = clock64();
    for (int i = 0; i < iters; i++) {
        asm volatile("mad.lo.cc.u32  %0, %4, %0, %1;\n\t"
                     "madc.lo.cc.u32 %1, %4, %1, %2;\n\t"
                     "madc.lo.cc.u32 %2, %4, %2, %3;\n\t"
                     "madc.lo.u32    %3, %4, %3, %0;" : "+r"(t0_), "+r"(t1_), "+r"(t2_), "+r"(t3_) : "r"(b));
    }
    long long t1 = clock64();
    out[0] = t0_ ^ t1_ ^ t2_ ^ t3_;
    cyc[0] = t1 - t0;
}


__global__ void k_mul_lat(const uint32_t* in, uint32_t* out, int iters, long long* cyc) {
    fe x = fq::load(in), y = fq::load(in + 8);
    long long t0 = clock64();
    for (int i = 0; i < iters; i++) x = fq::mul(x, y);
    long long t1 = clock64();
    fq::store(out, x);
    cyc[0] = t1 - t0;
}

template <bool SQR>
__global__ void k_mul_tput(const uint32_t* in, uint32_t* out, int iters) {
    fe x0 = fq::load(in), x1 = fq::load(in), y = fq::load(in + 8);
    x0.v[0] ^= threadIdx.x;
    x1.v[0] ^= threadIdx.x + 1;
    for (int i = 0; i < iters; i++) {
        x0 = SQR ? fq::sqr_fused(x0) : fq::mul(x0, y);
        x1 = SQR ? fq::sqr_fused(x1) : fq::mul(x1, y);
    }
    fq::store(out + 8 * (blockIdx.x * blockDim.x + threadIdx.x), fq::add(x0, x1));
}

__global__ void k_sqr_lat(const uint32_t* in, uint32_t* out, int iters, long long* cyc) {
    fe x = fq::load(in);
    long long t0 = clock64();
    for (int i = 0; i < iters; i++) x = fq::sqr_fused(x);
    long long t1 = clock64();
    fq::store(out, x);
    cyc[0] = t1 - t0;
}

int main() {
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, 0));
    int sms = prop.multiProcessorCount;
    printf("device %s, %d SMs\n", prop.name, sms);
    uint32_t *d_out, *d_in;
    long long* d_cyc;
    CK(cudaMalloc(&d_out, sizeof(uint32_t) * 8 * (size_t)(1 << 22)));
    CK(cudaMalloc(&d_in, sizeof(uint32_t) * 16));
    CK(cudaMalloc(&d_cyc, sizeof(long long)));
    uint32_t h_in[16];
    for (int i = 0; i < 16; i++) h_in[i] = 0x9e3779b9u * (i + 1);
    h_in[7] &= 0x0fffffffu;  // both operands below p
    h_in[15] &= 0x0fffffffu;
    CK(cudaMemcpy(d_in, h_in, sizeof(h_in), cudaMemcpyHostToDevice));
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float ms;
    long long cyc;
    const int blocks = sms * 8, tpb = 256, iters = 4096;
    double ops = (double)blocks * tpb * iters * 8;
    k_imad_tput<<<blocks, tpb>>>(d_out, 16, 1);
    cudaEventRecord(e0);
    k_imad_tput<<<blocks, tpb>>>(d_out, iters, 1);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("mad.lo.u32 throughput: %.3f Tops/s\n", ops / (ms * 1e-3) / 1e12);
    cudaEventRecord(e0);
    k_imadhi_tput<<<blocks, tpb>>>(d_out, iters, 1);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("mad.hi.u32 throughput: %.3f Tops/s\n", ops / (ms * 1e-3) / 1e12);
    cudaEventRecord(e0);
    k_madc_tput<<<blocks, tpb>>>(d_out, iters / 4, 1);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("madc.lo.cc chain throughput: %.3f Tops/s\n", (double)blocks * tpb * (iters / 4) * 32 / (ms * 1e-3) / 1e12);
    cudaEventRecord(e0);
    k_pair_row_tput<<<blocks, tpb>>>(d_out, iters / 4, 1);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("paired lo/hi rows: %.3f T full products/s\n", (double)blocks * tpb * (iters / 4) * 16 / (ms * 1e-3) / 1e12);
    cudaEventRecord(e0);
    k_unpaired_tput<<<blocks, tpb>>>(d_out, iters, 1);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("unpaired lo + hi: %.3f T pairs/s\n", (double)blocks * tpb * iters * 8 / (ms * 1e-3) / 1e12);
    k_imad_lat<<<1, 1>>>(d_out, iters, 3, d_cyc);
    CK(cudaMemcpy(&cyc, d_cyc, 8, cudaMemcpyDeviceToHost));
    printf("mad.lo dependent latency: %.2f cycles\n", (double)cyc / (iters * 4));
    k_madc_lat<<<1, 1>>>(d_out, iters, 3, d_cyc);
    CK(cudaMemcpy(&cyc, d_cyc, 8, cudaMemcpyDeviceToHost));
    printf("madc chain latency per instruction: %.2f cycles\n", (double)cyc / (iters * 4));
    k_mul_lat<<<1, 1>>>(d_in, d_out, 2000, d_cyc);
    CK(cudaMemcpy(&cyc, d_cyc, 8, cudaMemcpyDeviceToHost));
    printf("fq::mul latency: %.1f cycles\n", (double)cyc / 2000);
    const int mb = sms * 16, mt = 128, mit = 256;
    k_mul_tput<false><<<mb, mt>>>(d_in, d_out, 8);
    cudaEventRecord(e0);
    k_mul_tput<false><<<mb, mt>>>(d_in, d_out, mit);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    double muls = (double)mb * mt * mit * 2;
    printf("fq::mul throughput: %.2f Gmul/s = %.2f T IMAD slots/s (264 slots per mul)\n", muls / (ms * 1e-3) / 1e9,
           muls * 264 / (ms * 1e-3) / 1e12);
    cudaEventRecord(e0);
    k_mul_tput<true><<<mb, mt>>>(d_in, d_out, mit);
    cudaEventRecord(e1);
    CK(cudaEventSynchronize(e1));
    cudaEventElapsedTime(&ms, e0, e1);
    printf("fq::sqr_fused throughput: %.2f Gsqr/s = %.2f T IMAD slots/s (208 slots per squaring)\n",
           muls / (ms * 1e-3) / 1e9, muls * 208 / (ms * 1e-3) / 1e12);
    k_sqr_lat<<<1, 1>>>(d_in, d_out, 2000, d_cyc);
    CK(cudaMemcpy(&cyc, d_cyc, 8, cudaMemcpyDeviceToHost));
    printf("fq::sqr_fused latency: %.1f cycles\n", (double)cyc / 2000);
    CK(cudaGetLastError());
    return 0;
}
