// w4a4.cu -- a3: W4A4 linear (draft pass).
//
// QSPEC summary page, background terms: "W4A4" quantises weights and
// activations to 4 bits and runs a low-precision kernel with no
// dequantisation; the products are accumulated in INT32 and then scaled to a
// 16-bit result.  "QSPEC structure": the draft pass shares the verify pass's
// 4-bit weights.
//
// Bit-exact definition (shared with the CPU oracle, written separately):
//   I[m][n][g] = sum_{k in g} q[m][k] (W[n][k] - z[n][g])         exact int32
//             = sum_{k in g} q W  -  z qs[m][g]
//   acc = 0; for g ascending: acc = fmaf((float) I, sx[m][g] * s[n][g], acc)
//   y[m][n] = bf16_rn(acc)
//
// Small-M path (draft decode, M <= 8 tokens per CTA): CUDA-core dp4a.
//   - the CTA stages its tokens' INT4 activations in shared memory as signed
//     bytes, in the order the weight nibbles unpack to (even k / odd k);
//   - a quad of 4 lanes owns one (row, group) item: each lane loads 16 bytes
//     (32 weights), dp4a against the activations, two shuffles give the
//     group's integer sum; the quad leader stores I to shared memory;
//   - once every group of the CTA's 16 rows is in, one thread per
//     (row, token) folds the groups in ascending order in fp32.
// HBM-bound at small M: 0.5 byte of weight + 4/128 byte of scale/zero per
// weight.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {

constexpr int kThreads = 256;
constexpr int kQuads = kThreads / 4;
constexpr int kRows = 16;           // output rows per CTA
constexpr int kPrefetch = 8;        // items in flight per quad

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// smem layout: acts int2 [MT][K/8] (.x: q of k0,k2,k4,k6 ; .y: k1,k3,k5,k7 as
// signed bytes), I int32 [G][kRows][MT], s float [G][kRows], sx float [MT][G],
// qs int [MT][G].
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
    w4a4_gemv_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ sx,
                     const int32_t *__restrict__ qs, const uint8_t *__restrict__ packed,
                     const uint32_t *__restrict__ sz, int M, int N, int K,
                     uint16_t *__restrict__ y, int ldy, int32_t *__restrict__ dbg_I) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = K / kGroup;
    const int K8 = K / 8;
    int2 *acts = reinterpret_cast<int2 *>(smem_raw);
    int32_t *ibuf = reinterpret_cast<int32_t *>(acts + (size_t)MT * K8);
    float *sbuf = reinterpret_cast<float *>(ibuf + kRows * MT * G);
    float *sxs = sbuf + kRows * G;
    int32_t *qss = reinterpret_cast<int32_t *>(sxs + MT * G);

    const int tok0 = blockIdx.y * MT;
    const int row0 = blockIdx.x * kRows;
    const int quad = threadIdx.x >> 2, qc = threadIdx.x & 3;
    const int n_items = kRows * G;
    const size_t row_u4 = (size_t)K / 32;   // uint4 per packed row
    const uint4 *wbase = reinterpret_cast<const uint4 *>(packed);

    pdl_launch_dependents();
    // weights and scale words are immutable: start streaming them before the
    // previous kernel has finished
    uint4 ring[kPrefetch];
    uint32_t ring_sz[kPrefetch];
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p) {
        int it = quad + p * kQuads;
        int r = it / G, g = it % G, n = row0 + r;
        if (it < n_items && n < N) {
            ring[p] = ldg_stream(wbase + (size_t)n * row_u4 + g * 4 + qc);
            ring_sz[p] = __ldg(sz + (size_t)n * G + g);
        }
    }
    pdl_wait();

    // stage activations: nibbles -> signed bytes, even-k and odd-k words
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(xq);
    for (int i = threadIdx.x; i < MT * K8; i += kThreads) {
        int t = i / K8, j = i % K8, m = tok0 + t;
        uint32_t w = m < M ? xw[(size_t)m * K8 + j] : 0u;
        uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        // two's-complement nibble -> byte: (v ^ 8) - 8, per byte without borrows
        lo = __vsub4(lo ^ 0x08080808u, 0x08080808u);
        hi = __vsub4(hi ^ 0x08080808u, 0x08080808u);
        acts[i] = make_int2((int)lo, (int)hi);
    }
    for (int i = threadIdx.x; i < MT * G; i += kThreads) {
        int t = i / G, m = tok0 + t;
        sxs[i] = m < M ? sx[(size_t)m * G + i % G] : 0.0f;
        qss[i] = m < M ? qs[(size_t)m * G + i % G] : 0;
    }
    __syncthreads();

    // phase 1: group integers of the CTA's rows
    for (int base = quad; base < n_items; base += kPrefetch * kQuads) {
#pragma unroll
        for (int p = 0; p < kPrefetch; ++p) {
            const int it = base + p * kQuads;
            if (it >= n_items) break;
            const int r = it / G, g = it % G;
            const uint4 wv = ring[p];
            const uint32_t szw = ring_sz[p];
            {
                int itn = it + kPrefetch * kQuads;
                int rn = itn / G, gn = itn % G, nn = row0 + rn;
                if (itn < n_items && nn < N) {
                    ring[p] = ldg_stream(wbase + (size_t)nn * row_u4 + gn * 4 + qc);
                    ring_sz[p] = __ldg(sz + (size_t)nn * G + gn);
                }
            }
            const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t wl[4], wh[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wl[u] = w[u] & 0x0F0F0F0Fu;
                wh[u] = (w[u] >> 4) & 0x0F0F0F0Fu;
            }
            const int zi = (int)__half2float(__ushort_as_half((uint16_t)(szw >> 16)));
            if (qc == 0) sbuf[g * kRows + r] = __half2float(__ushort_as_half((uint16_t)(szw & 0xFFFF)));
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int4 *ap = reinterpret_cast<const int4 *>(acts + (size_t)t * K8 + g * 16 + qc * 4);
                int4 a01 = ap[0], a23 = ap[1];
                int s = 0;
                s = __dp4a(a01.x, (int)wl[0], s);
                s = __dp4a(a01.y, (int)wh[0], s);
                s = __dp4a(a01.z, (int)wl[1], s);
                s = __dp4a(a01.w, (int)wh[1], s);
                s = __dp4a(a23.x, (int)wl[2], s);
                s = __dp4a(a23.y, (int)wh[2], s);
                s = __dp4a(a23.z, (int)wl[3], s);
                s = __dp4a(a23.w, (int)wh[3], s);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (qc == 0) ibuf[(g * kRows + r) * MT + t] = s - zi * qss[t * G + g];
            }
        }
    }
    __syncthreads();

    // phase 2: fold the groups in ascending order, one thread per (row, token);
    // shared memory only
    for (int p = threadIdx.x; p < kRows * MT; p += kThreads) {
        const int r = p / MT, t = p % MT, n = row0 + r, m = tok0 + t;
        if (n >= N || m >= M) continue;
        float acc = 0.0f;
        for (int g = 0; g < G; ++g) {
            const int32_t I = ibuf[(g * kRows + r) * MT + t];
            const float c = __fmul_rn(sxs[t * G + g], sbuf[g * kRows + r]);
            acc = __fmaf_rn(__int2float_rn(I), c, acc);
            if (dbg_I) dbg_I[((size_t)m * N + n) * G + g] = I;
        }
        y[(size_t)m * ldy + n] = float_to_bf16_bits(acc);
    }
}

template <int MT>
size_t gemv_smem_bytes(int K) {
    const int G = K / kGroup;
    return (size_t)MT * (K / 8) * sizeof(int2) + (size_t)kRows * MT * G * 4 + (size_t)kRows * G * 4 +
           (size_t)MT * G * 8;
}

constexpr size_t kMaxSmem = 200 * 1024;

template <int MT>
int launch_gemv(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I,
                cudaStream_t st) {
    size_t smem = gemv_smem_bytes<MT>(K);
    int rc = smem_limit_once(reinterpret_cast<const void *>(&w4a4_gemv_kernel<MT>), MT, (int)kMaxSmem);
    if (rc) return rc;
    dim3 grid((unsigned)((N + kRows - 1) / kRows), (unsigned)((M + MT - 1) / MT));
    return launch_pdl("qspec_linear_w4a4", w4a4_gemv_kernel<MT>, grid, dim3(kThreads), smem, st, xq, sx,
                      qs, packed, sz, M, N, K, y, ldy, dbg_I);
}

}  // namespace

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_linear_w4a4(const uint8_t *xq, const float *sx, const int32_t *qs,
                                 const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                                 uint16_t *y_bf16, int ldy, int32_t *dbg_I, int32_t *dev_status,
                                 qspec_stream_t stream) {
    if (!xq || !sx || !qs || !packed || !sz || !y_bf16) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < kGroup || K % kGroup || ldy < N) return QSPEC_ERR_SHAPE;
    if (!aligned(xq, 16) || !aligned(packed, 16) || !aligned(sz, 4) || !aligned(sx, 4) ||
        !aligned(qs, 4) || !aligned(y_bf16, 2) || (dbg_I && !aligned(dbg_I, 4)))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    if (M > 8) return launch_w4a4_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st);
    if (M == 1 && gemv_smem_bytes<1>(K) <= kMaxSmem)
        return launch_gemv<1>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (M <= 2 && gemv_smem_bytes<2>(K) <= kMaxSmem)
        return launch_gemv<2>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (M <= 4 && gemv_smem_bytes<4>(K) <= kMaxSmem)
        return launch_gemv<4>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (gemv_smem_bytes<8>(K) <= kMaxSmem)
        return launch_gemv<8>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (gemv_smem_bytes<4>(K) <= kMaxSmem)
        return launch_gemv<4>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    return QSPEC_ERR_SHAPE;
}
