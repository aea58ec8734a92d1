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
// Small-M path (M <= 32, draft decode): FP8 warp MMA on exact small
// integers, described below.  Larger M: tcgen05 (w4a4_tc.cu).
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {

// ---------------------------------------------------------------------------
// Small-M path on the FP8 tensor cores (warp MMA m16n8k32, e4m3 operands).
//
// An E4M3 byte holding a value b in 0..15 is exactly b * 2^-9 (subnormals for
// b < 8, exponent 1 above), so the unpacked nibbles feed the MMA with no table:
//   A (weights): codes c, one byte each            -> c * 2^-9
//   B (tokens):  u = q + 8 = nibble ^ 8, one byte   -> u * 2^-9
//   B column OC: all ones                           -> 2^-9
// and the fp32 accumulator of one 128-wide group holds, exactly,
//   D = sum u c * 2^-18   and   C = sum c * 2^-18 (column OC).
// Then I = sum q (c - z) = sum u c - 8 sum c - z qs, all integers below 2^15:
//   I = fmaf(-z, qs, fmaf(D, 2^18, -8 C 2^18)) exactly in fp32.
// Each thread loads 16 bytes (32 codes) of two rows per group; the k order
// inside the MMA is permuted identically on A and B (even k then odd k of
// every 8), so unpacking is two logic operations per word.  Warps split the
// groups of a 16-row tile; one thread per (row, token) folds in order.
// ---------------------------------------------------------------------------
namespace mmak {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kPrefetch = 4;           // groups in flight per warp

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Persistent over 16-row tiles.  smem: actf uint2 [MT][G][16] (B fragments),
// I float [2][G][16][MT] (double buffer), s float [2][G][16], sx float [MT][G],
// qs float [MT][G].  Warp w owns groups w, w + 8, ...; per warp the (tile,
// group) items form one sequence, so the prefetch ring runs across tiles.
// After a tile, one warp folds it (ascending groups) while the others start
// the next tile; the next barrier orders the fold before its buffer is reused.
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
    w4a4_mma_gemv_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ sx,
                         const int32_t *__restrict__ qs, const uint8_t *__restrict__ packed,
                         const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y, int ldy,
                         int32_t *__restrict__ dbg_I) {
    constexpr int OC = MT == 1 ? 1 : 7;          // the all-ones B column
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = K / kGroup;
    uint2 *actf = reinterpret_cast<uint2 *>(smem_raw);
    float *ibuf = reinterpret_cast<float *>(actf + (size_t)MT * G * 16);
    float *sbuf = ibuf + (size_t)2 * G * 16 * MT;
    float *sxs = sbuf + (size_t)2 * G * 16;
    float *qss = sxs + (size_t)MT * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qr = lane >> 2, qc = lane & 3;
    const int tok0 = blockIdx.y * MT;
    const int n_tiles = (N + 15) / 16;
    const size_t row_u4 = (size_t)K / 32;
    const uint4 *wbase = reinterpret_cast<const uint4 *>(packed) + qc;
    const int ng = warp < G ? (G - warp + kWarps - 1) / kWarps : 0;     // this warp's groups per tile
    const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int n_items = ng * my_tiles;

    // item cursor -> (tile, group); advanced incrementally, no division
    struct Cursor {
        int step, gi;
    };
    auto load_item = [&](const Cursor &c, uint4 &wa, uint4 &wb, uint32_t &za, uint32_t &zb) {
        const int tile = blockIdx.x + c.step * gridDim.x, g = warp + c.gi * kWarps;
        const int r0 = tile * 16 + qr, r1 = r0 + 8;
        const bool v0 = r0 < N, v1 = r1 < N;
        wa = __ldg(wbase + (size_t)(v0 ? r0 : 0) * row_u4 + g * 4);
        wb = __ldg(wbase + (size_t)(v1 ? r1 : 0) * row_u4 + g * 4);
        za = v0 ? __ldg(sz + (size_t)r0 * G + g) : 0u;
        zb = v1 ? __ldg(sz + (size_t)r1 * G + g) : 0u;
    };
    auto advance = [&](Cursor &c) {
        if (++c.gi == ng) {
            c.gi = 0;
            ++c.step;
        }
    };

    pdl_launch_dependents();
    // immutable weights and scale words first
    uint4 ra[kPrefetch], rb[kPrefetch];
    uint32_t sa[kPrefetch], sb[kPrefetch];
    Cursor pc = {0, 0};
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p) {
        if (p < n_items) {
            load_item(pc, ra[p], rb[p], sa[p], sb[p]);
            advance(pc);
        }
    }
    pdl_wait();

    // this CTA's tokens, once: B fragments (u = q + 8 as bytes, even k then odd k), sx, qs
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(xq);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int m = tok0 + t;
        for (int i = threadIdx.x; i < G * 16; i += kThreads) {
            const uint32_t w = m < M ? xw[(size_t)m * (K / 8) + i] ^ 0x88888888u : 0u;
            actf[(size_t)t * G * 16 + i] = make_uint2(w & 0x0F0F0F0Fu, (w >> 4) & 0x0F0F0F0Fu);
        }
        for (int g = threadIdx.x; g < G; g += kThreads) {
            sxs[t * G + g] = m < M ? sx[(size_t)m * G + g] : 0.0f;
            qss[t * G + g] = m < M ? (float)qs[(size_t)m * G + g] : 0.0f;
        }
    }
    __syncthreads();

    const bool tok_row = qr < MT && tok0 + qr < M;     // this thread feeds a real token column
    const int tq = qr < MT ? qr : 0;
    const float two18 = 262144.0f;

    // end of tile `step`: every warp arrives once per tile; then one warp folds it
    auto tile_done = [&](int step) {
        __syncthreads();
        if (warp != (step & (kWarps - 1))) return;
        const int tile = blockIdx.x + step * gridDim.x;
        const float *ib = ibuf + (size_t)(step & 1) * G * 16 * MT;
        const float *sbb = sbuf + (size_t)(step & 1) * G * 16;
        for (int p = lane; p < 16 * MT; p += 32) {
            const int r = p / MT, t = p - (p / MT) * MT, n = tile * 16 + r, m = tok0 + t;
            if (n >= N || m >= M) continue;
            float acc = 0.0f;
            for (int g = 0; g < G; ++g) {
                const float I = ib[((size_t)g * 16 + r) * MT + t];
                acc = __fmaf_rn(I, __fmul_rn(sxs[t * G + g], sbb[(size_t)g * 16 + r]), acc);
                if (dbg_I) dbg_I[((size_t)m * N + n) * G + g] = (int32_t)I;
            }
            y[(size_t)m * ldy + n] = float_to_bf16_bits(acc);
        }
    };

    Cursor cc = {0, 0};
    int cur = 0;                                          // tile step being produced
    for (int base = 0; base < n_items; base += kPrefetch) {
#pragma unroll
        for (int p = 0; p < kPrefetch; ++p) {
            const int it = base + p;
            if (it >= n_items) break;
            if (cc.step != cur) {                         // this warp's first item of the next tile
                tile_done(cur);
                cur = cc.step;
            }
            const int g = warp + cc.gi * kWarps;
            float *ib = ibuf + (size_t)(cur & 1) * G * 16 * MT;
            float *sbb = sbuf + (size_t)(cur & 1) * G * 16;
            const uint4 wa = ra[p], wb = rb[p];
            const uint32_t za = sa[p], zb = sb[p];
            if (it + kPrefetch < n_items) {
                load_item(pc, ra[p], rb[p], sa[p], sb[p]);
                advance(pc);
            }
            uint32_t bf0[4], bf1[4];
            if (tok_row) {
                const uint4 *ap = reinterpret_cast<const uint4 *>(actf + ((size_t)tq * G + g) * 16 + qc * 4);
                const uint4 f01 = ap[0], f23 = ap[1];
                bf0[0] = f01.x; bf1[0] = f01.y; bf0[1] = f01.z; bf1[1] = f01.w;
                bf0[2] = f23.x; bf1[2] = f23.y; bf0[3] = f23.z; bf1[3] = f23.w;
            } else {
                const uint32_t one = qr == OC ? 0x01010101u : 0u;
#pragma unroll
                for (int j = 0; j < 4; ++j) bf0[j] = bf1[j] = one;
            }
            const uint32_t wa_[4] = {wa.x, wa.y, wa.z, wa.w}, wb_[4] = {wb.x, wb.y, wb.z, wb.w};
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mma_e4m3_16832(d, wa_[j] & 0x0F0F0F0Fu, wb_[j] & 0x0F0F0F0Fu, (wa_[j] >> 4) & 0x0F0F0F0Fu,
                               (wb_[j] >> 4) & 0x0F0F0F0Fu, bf0[j], bf1[j]);
            // D: rows (qr, qr + 8) x columns (2 qc, 2 qc + 1); C from column OC
            float c_a, c_b;
            if (MT == 1) {
                c_a = d[1];
                c_b = d[3];
            } else {
                c_a = __shfl_sync(0xffffffffu, d[1], (lane & ~3) | 3);
                c_b = __shfl_sync(0xffffffffu, d[3], (lane & ~3) | 3);
            }
            if (2 * qc < MT) {
                const float ia = c_a * (-8.0f * two18), ibv = c_b * (-8.0f * two18);   // exact
                const float zfa = __half2float(__ushort_as_half((uint16_t)(za >> 16)));
                const float zfb = __half2float(__ushort_as_half((uint16_t)(zb >> 16)));
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * qc + e;
                    if (t < MT && t != OC) {
                        const float q_s = qss[t * G + g];
                        ib[((size_t)g * 16 + qr) * MT + t] = __fmaf_rn(-zfa, q_s, __fmaf_rn(d[e], two18, ia));
                        ib[((size_t)g * 16 + qr + 8) * MT + t] = __fmaf_rn(-zfb, q_s, __fmaf_rn(d[2 + e], two18, ibv));
                    }
                }
            }
            if (qc == 0) {
                sbb[(size_t)g * 16 + qr] = __half2float(__ushort_as_half((uint16_t)(za & 0xFFFF)));
                sbb[(size_t)g * 16 + qr + 8] = __half2float(__ushort_as_half((uint16_t)(zb & 0xFFFF)));
            }
            advance(cc);
        }
    }
    // the last tile with items, then the remaining ones (warps without groups)
    for (; cur < my_tiles; ++cur) tile_done(cur);
}

template <int MT>
size_t smem_bytes(int K) {
    const int G = K / kGroup;
    return (size_t)MT * G * 16 * sizeof(uint2) + (size_t)2 * G * 16 * MT * 4 + (size_t)2 * G * 16 * 4 +
           (size_t)MT * G * 8;
}

template <int MT>
int launch(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed, const uint32_t *sz, int M,
           int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, cudaStream_t st) {
    const size_t smem = smem_bytes<MT>(K);
    int rc = smem_limit_once(reinterpret_cast<const void *>(&w4a4_mma_gemv_kernel<MT>), 8 + MT, 200 * 1024);
    if (rc) return rc;
    const int n_tiles = (N + 15) / 16, token_tiles = (M + MT - 1) / MT;
    const int per_col = std::max(1, 2 * sm_count() / token_tiles);
    dim3 grid((unsigned)std::min(n_tiles, per_col), (unsigned)token_tiles);
    return launch_pdl("qspec_linear_w4a4", w4a4_mma_gemv_kernel<MT>, grid, dim3(kThreads), smem, st, xq, sx, qs,
                      packed, sz, M, N, K, y, ldy, dbg_I);
}

}  // namespace mmak

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
    if (M > 32) return launch_w4a4_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st);
    constexpr size_t kMaxSmem = 200 * 1024;
    if (M == 1 && mmak::smem_bytes<1>(K) <= kMaxSmem)
        return mmak::launch<1>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (M == 2 && mmak::smem_bytes<2>(K) <= kMaxSmem)
        return mmak::launch<2>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (M <= 4 && mmak::smem_bytes<4>(K) <= kMaxSmem)
        return mmak::launch<4>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (mmak::smem_bytes<7>(K) <= kMaxSmem)
        return mmak::launch<7>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (mmak::smem_bytes<4>(K) <= kMaxSmem)
        return mmak::launch<4>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    if (mmak::smem_bytes<1>(K) <= kMaxSmem)
        return mmak::launch<1>(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, st);
    return QSPEC_ERR_SHAPE;
}
