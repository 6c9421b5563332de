// Host build of the scalar split in glv.cuh, for the CPU tests: reads scalars
// (8 hex limbs, little-endian, one scalar per line, already < r) on stdin and
// prints "s1 |k1| s2 |k2|" per line (signs 0/1, magnitudes in hex).
#define __host__
#define __device__
#define __forceinline__ inline
#include <cstdio>

#include "glv.cuh"

int main() {
    uint32_t k[8];
    while (scanf("%x %x %x %x %x %x %x %x", &k[0], &k[1], &k[2], &k[3], &k[4], &k[5], &k[6], &k[7]) == 8) {
        uint32_t k1[4], k2[4], s1, s2;
        glv::split(k, k1, k2, s1, s2);
        printf("%u %08x%08x%08x%08x %u %08x%08x%08x%08x\n", s1, k1[3], k1[2], k1[1], k1[0], s2, k2[3], k2[2], k2[1],
               k2[0]);
    }
    return 0;
}
