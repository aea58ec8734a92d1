// w4a16.cu -- a4: W4A16 linear, y = x W^T with W^ = s (W - z), fp32
// accumulation, bf16 output.
//
// QSPEC summary page, background terms: "W4A16" stores weights in 4 bits and
// keeps 16-bit activations, dequantising the weights for the matmul,
// W^ = s (W_INT4 - z); "QSPEC structure": the verify pass over the gamma + 1
// candidate rows of every sequence.
//
// Small-M path (decode verify, M = B (gamma + 1) <= 16 per token tile): warp
// MMA m16n8k16 bf16 with fp32 accumulation.  The weight tile is the MMA's A
// operand (16 output channels x 16 k), the activations its B operand (16 k x 8
// tokens).  Dequantisation happens in registers and is split so the tensor
// core sees exact small integers:
//   - a code c becomes the bf16 value 128 + c by OR-ing it into the mantissa
//     of 128.0 (bits 0x4300 | c); no conversion instruction is needed;
//   - per group g, D = sum_k (128 + c_k) x_k is accumulated by the MMA, and the
//     epilogue applies y += s_g (D - (128 + z_g) X_g), X_g = sum_{k in g} x_k,
//     which equals sum_k s_g (c_k - z_g) x_k, the definition.
// The k order inside the MMA is permuted identically on A and B so that each
// thread's 16-byte weight load and 16-byte activation loads feed its fragments
// without shuffles (a dot product does not depend on the k order).
//
// HBM-bound for M <= 16: 0.5 byte of weight + 4/128 byte of scale/zero per
// weight dominates; each CTA streams 16-row tiles, split over its 8 warps by
// group, with a 4-group prefetch per warp.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ void mma_bf16_16816(float &d0, float &d1, float &d2, float &d3,
                                               uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Eight codes of one 32-bit word (k0..k7 in nibbles 0..7) -> four bf16x2 of
// (128 + c): (k0,k4), (k1,k5), (k2,k6), (k3,k7).
__device__ __forceinline__ void codes_to_bf16x2(uint32_t w, uint32_t p[4]) {
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
    p[0] = (w & mask) | magic;
    p[1] = ((w >> 4) & mask) | magic;
    p[2] = ((w >> 8) & mask) | magic;
    p[3] = ((w >> 12) & mask) | magic;
}

// Eight bf16 activations x0..x7 (four 32-bit words) -> the same pairing.
__device__ __forceinline__ void acts_to_pairs(uint4 v, uint32_t p[4]) {
    p[0] = __byte_perm(v.x, v.z, 0x5410);
    p[1] = __byte_perm(v.x, v.z, 0x7632);
    p[2] = __byte_perm(v.y, v.w, 0x5410);
    p[3] = __byte_perm(v.y, v.w, 0x7632);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// NT token tiles of 8 per CTA (NT = 1 or 2).  grid.x: persistent over 16-row
// tiles; grid.y: token tiles of 8 * NT.
template <int NT>
__global__ void __launch_bounds__(kThreads, 2)
    w4a16_mma_kernel(const uint16_t *__restrict__ x, int ldx, const uint8_t *__restrict__ packed,
                     const uint32_t *__restrict__ sz, int M, int N, int K,
                     uint16_t *__restrict__ y, int ldy) {
    extern __shared__ float smem[];
    const int G = K / kGroup;
    float *xg = smem;                                   // [NT*8][G]   group sums of x
    float *red = smem + NT * 8 * G;                     // [kWarps][NT*8][16]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qr = lane >> 2, qc = lane & 3;
    const int tok0 = blockIdx.y * 8 * NT;
    const int n_tiles = (N + 15) / 16;
    const size_t row_bytes = (size_t)K / 2;
    constexpr int kPrefetch = NT == 1 ? 4 : 2;   // groups in flight per warp

    pdl_launch_dependents();
    // prefetch ring over this warp's groups g = warp, warp + 8, ... of the
    // first tile: weights are immutable, so this overlaps the previous kernel
    uint4 ring0[kPrefetch], ring1[kPrefetch];
    {
        const int tile = blockIdx.x;
        const int r0 = tile * 16 + qr, r1 = r0 + 8;
        const uint4 *w0p = reinterpret_cast<const uint4 *>(packed + (size_t)(r0 < N ? r0 : 0) * row_bytes) + qc;
        const uint4 *w1p = reinterpret_cast<const uint4 *>(packed + (size_t)(r1 < N ? r1 : 0) * row_bytes) + qc;
#pragma unroll
        for (int j = 0; j < kPrefetch; ++j) {
            int g = warp + j * kWarps;
            if (tile < n_tiles && g < G) {
                ring0[j] = ldg_stream(w0p + g * 4);
                ring1[j] = ldg_stream(w1p + g * 4);
            }
        }
    }
    pdl_wait();

    // group sums X_g of this CTA's tokens, one (token, group) per thread at a time
    for (int i = threadIdx.x; i < NT * 8 * G; i += kThreads) {
        const int t = i / G, g = i % G, m = tok0 + t;
        float s = 0.0f;
        if (m < M) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(x + (size_t)m * ldx + (size_t)g * kGroup);
            uint4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = __ldg(xp + u);
            float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                part[0] += __uint_as_float(v[u].x << 16) + __uint_as_float(v[u].x & 0xFFFF0000u);
                part[1] += __uint_as_float(v[u].y << 16) + __uint_as_float(v[u].y & 0xFFFF0000u);
                part[2] += __uint_as_float(v[u].z << 16) + __uint_as_float(v[u].z & 0xFFFF0000u);
                part[3] += __uint_as_float(v[u].w << 16) + __uint_as_float(v[u].w & 0xFFFF0000u);
            }
            s = (part[0] + part[1]) + (part[2] + part[3]);
        }
        xg[t * G + g] = s;
    }
    __syncthreads();

    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int r0 = tile * 16 + qr, r1 = r0 + 8;
        const bool v0 = r0 < N, v1 = r1 < N;
        const uint4 *w0p = reinterpret_cast<const uint4 *>(packed + (size_t)(v0 ? r0 : 0) * row_bytes) + qc;
        const uint4 *w1p = reinterpret_cast<const uint4 *>(packed + (size_t)(v1 ? r1 : 0) * row_bytes) + qc;

        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

        if (tile != (int)blockIdx.x) {
#pragma unroll
            for (int j = 0; j < kPrefetch; ++j) {
                int g = warp + j * kWarps;
                if (g < G) {
                    ring0[j] = ldg_stream(w0p + g * 4);
                    ring1[j] = ldg_stream(w1p + g * 4);
                }
            }
        }
        // activation fragments of the warp's first group
        uint4 xv[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int m = tok0 + nt * 8 + qr;
            const uint4 *xp = reinterpret_cast<const uint4 *>(
                x + (size_t)(m < M ? m : 0) * ldx + (size_t)warp * kGroup + qc * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                xv[nt][u] = (m < M && warp < G) ? __ldg(xp + u) : make_uint4(0, 0, 0, 0);
        }
        for (int gb = warp; gb < G; gb += kPrefetch * kWarps) {
#pragma unroll
            for (int slot = 0; slot < kPrefetch; ++slot) {
                const int g = gb + slot * kWarps;
                if (g >= G) break;
                uint4 wa = ring0[slot], wb = ring1[slot];
                {
                    int gn = g + kPrefetch * kWarps;
                    if (gn < G) {
                        ring0[slot] = ldg_stream(w0p + gn * 4);
                        ring1[slot] = ldg_stream(w1p + gn * 4);
                    }
                }
                // next group's activation fragments
                uint4 xn[NT][4];
                const int gx = g + kWarps;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m = tok0 + nt * 8 + qr;
                    const uint4 *xp = reinterpret_cast<const uint4 *>(
                        x + (size_t)(m < M ? m : 0) * ldx + (size_t)(gx < G ? gx : 0) * kGroup + qc * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        xn[nt][u] = (m < M && gx < G) ? __ldg(xp + u) : make_uint4(0, 0, 0, 0);
                }
                const uint32_t wr0[4] = {wa.x, wa.y, wa.z, wa.w};
                const uint32_t wr1[4] = {wb.x, wb.y, wb.z, wb.w};

                // this group's scale and zero point for rows r0, r1
                uint32_t sz0 = v0 ? __ldg(sz + (size_t)r0 * G + g) : 0u;
                uint32_t sz1 = v1 ? __ldg(sz + (size_t)r1 * G + g) : 0u;
                float s0 = __half2float(__ushort_as_half((uint16_t)(sz0 & 0xFFFF)));
                float s1 = __half2float(__ushort_as_half((uint16_t)(sz1 & 0xFFFF)));
                float o0 = 128.0f + __half2float(__ushort_as_half((uint16_t)(sz0 >> 16)));
                float o1 = 128.0f + __half2float(__ushort_as_half((uint16_t)(sz1 >> 16)));

#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t pa0[4], pa1[4], pb[4];
                        codes_to_bf16x2(wr0[u], pa0);
                        codes_to_bf16x2(wr1[u], pa1);
                        acts_to_pairs(xv[nt][u], pb);
                        mma_bf16_16816(d[0], d[1], d[2], d[3], pa0[0], pa1[0], pa0[1], pa1[1], pb[0], pb[1]);
                        mma_bf16_16816(d[0], d[1], d[2], d[3], pa0[2], pa1[2], pa0[3], pa1[3], pb[2], pb[3]);
                    }
                    // D holds rows (qr, qr+8) x tokens (2qc, 2qc+1) of this tile
                    const float X0 = xg[(nt * 8 + 2 * qc) * G + g];
                    const float X1 = xg[(nt * 8 + 2 * qc + 1) * G + g];
                    acc[nt][0] = __fmaf_rn(s0, __fmaf_rn(-o0, X0, d[0]), acc[nt][0]);
                    acc[nt][1] = __fmaf_rn(s0, __fmaf_rn(-o0, X1, d[1]), acc[nt][1]);
                    acc[nt][2] = __fmaf_rn(s1, __fmaf_rn(-o1, X0, d[2]), acc[nt][2]);
                    acc[nt][3] = __fmaf_rn(s1, __fmaf_rn(-o1, X1, d[3]), acc[nt][3]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int u = 0; u < 4; ++u) xv[nt][u] = xn[nt][u];
            }
        }

        // reduce the 8 warps' partial sums and store bf16
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float *rw = red + (size_t)warp * NT * 8 * 16;
            rw[(nt * 8 + 2 * qc) * 16 + qr] = acc[nt][0];
            rw[(nt * 8 + 2 * qc + 1) * 16 + qr] = acc[nt][1];
            rw[(nt * 8 + 2 * qc) * 16 + qr + 8] = acc[nt][2];
            rw[(nt * 8 + 2 * qc + 1) * 16 + qr + 8] = acc[nt][3];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < NT * 8 * 16; i += kThreads) {
            int t = i / 16, r = i % 16;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += red[(size_t)w * NT * 8 * 16 + i];
            int m = tok0 + t, n = tile * 16 + r;
            if (m < M && n < N) y[(size_t)m * ldy + n] = float_to_bf16_bits(sum);
        }
        __syncthreads();
    }
}

template <int NT>
int launch_w4a16(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N,
                 int K, uint16_t *y, int ldy, cudaStream_t st) {
    const int G = K / kGroup;
    size_t smem = (size_t)(NT * 8 * G + kWarps * NT * 8 * 16) * sizeof(float);
    if (smem > 48 * 1024) return QSPEC_ERR_SHAPE;   // K up to ~90k
    const int n_tiles = (N + 15) / 16;
    const int token_tiles = (M + 8 * NT - 1) / (8 * NT);
    int per_col = std::max(1, 2 * sm_count() / token_tiles);
    dim3 grid((unsigned)std::min(n_tiles, per_col), (unsigned)token_tiles);
    return launch_pdl("qspec_linear_w4a16", w4a16_mma_kernel<NT>, grid, dim3(kThreads), smem, st, x, ldx,
                      packed, sz, M, N, K, y, ldy);
}

}  // namespace

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_linear_w4a16(const uint16_t *x_bf16, int ldx, const uint8_t *packed,
                                  const uint32_t *sz, int M, int N, int K, uint16_t *y_bf16,
                                  int ldy, int32_t *dev_status, qspec_stream_t stream) {
    if (!x_bf16 || !packed || !sz || !y_bf16) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < kGroup || K % kGroup || ldx < K || ldy < N) return QSPEC_ERR_SHAPE;
    if (!aligned(x_bf16, 16) || ldx % 8 || !aligned(packed, 16) || !aligned(sz, 4) ||
        !aligned(y_bf16, 2))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    if (M <= 8) return launch_w4a16<1>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, st);
    if (M <= 16) return launch_w4a16<2>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, st);
    return launch_w4a16_tc(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, dev_status, st);
}
