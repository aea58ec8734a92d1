// Exhaustive check of the library's group quantiser (quant_group<1>, the
// routine every quantising kernel calls) against its definition, q =
// clamp(rint(x / sx), -7, 7) with sx = amax / 7 by the IEEE division: for
// every bf16 amax > 0 (finite) and every bf16 x with |x| <= amax, the code of
// x in a group whose largest magnitude is amax.  Prints the number of pairs,
// code mismatches and scale mismatches.
#include <cstdio>

#include "qspec_device.cuh"

using namespace qspec;

__global__ void check(unsigned long long *cnt) {
    const uint32_t ab = blockIdx.x + 1;                          // amax bits 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(ab << 16);
    const float sx_ref = __fdiv_rn(amax, 7.0f);
    const int n_x = 2 * (int)(ab + 1);                           // magnitudes 0..ab, both signs
    const int n_groups = (n_x + 126) / 127;                      // slot 0 of a group holds amax
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    unsigned long long bad_q = 0, bad_s = 0, pairs = 0;
    for (int g0 = 2 * warp; g0 < n_groups; g0 += 2 * (blockDim.x >> 5)) {
        const int g = g0 + half;                                 // warp-uniform loop, lanes past the end idle
        uint32_t w[4];
        float xs[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int slot = 8 * hl + i, j = g * 127 + slot - 1;
            uint32_t b = 0;
            if (slot == 0) b = ab;
            else if (g < n_groups && j < n_x) b = (uint32_t)(j >> 1) | ((j & 1) ? 0x8000u : 0u);
            xs[i] = __uint_as_float(b << 16);
            if (i & 1) w[i >> 1] |= b << 16;
            else w[i >> 1] = b;
        }
        const uint4 v[1] = {make_uint4(w[0], w[1], w[2], w[3])};
        float scale;
        int qsum;
        bool bad = false;
        uint32_t nib[1];
        quant_group<1>(v, scale, qsum, bad, nib);
        if (g < n_groups) {
            if (hl == 0 && __float_as_uint(scale) != __float_as_uint(sx_ref)) ++bad_s;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int slot = 8 * hl + i, j = g * 127 + slot - 1;
                if (slot == 0 || j >= n_x) continue;
                const int ref = sx_ref != 0.0f ? max(-7, min(7, (int)rintf(__fdiv_rn(xs[i], sx_ref)))) : 0;
                const int got = (int)((int32_t)(nib[0] << (28 - 4 * i)) >> 28);
                bad_q += got != ref;
                ++pairs;
            }
        }
    }
    atomicAdd(cnt + 0, pairs);
    atomicAdd(cnt + 1, bad_q);
    atomicAdd(cnt + 2, bad_s);
}

int main() {
    unsigned long long *c = nullptr, h[3] = {0, 0, 0};
    if (cudaMalloc(&c, sizeof(h)) != cudaSuccess) return 2;
    cudaMemset(c, 0, sizeof(h));
    check<<<0x7F7F, 256>>>(c);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(h, c, sizeof(h), cudaMemcpyDeviceToHost);
    printf("pairs %llu code_mismatches %llu scale_mismatches %llu status %s\n", h[0], h[1], h[2], cudaGetErrorString(e));
    return e == cudaSuccess ? 0 : 1;
}
