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
// One token (the B = 1 draft decode): byte dot products (w4a4_dp4a.cu).
// Small M (2..32): f16 warp MMA on exact small integers, described below;
// 3 <= M <= 16 with at least one 128-row tile per SM: tensor-memory GEMV
// (w4a4_gemv_tc.cu).  Larger M: tcgen05 (w4a4_tc.cu).
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {

// ---------------------------------------------------------------------------
// Small-M path: warp MMA m16n8k16 with f16 operands and fp32 accumulation.
//
// OR-ing a code into the mantissa of the f16 value 1024 (bits 0x6400) gives
// 1024 + c exactly when the code sits in bits 0..3 of a half, and 1024 + 16 c
// when it sits in bits 4..7, so one logic operation turns a weight word (codes
// c0..c7 in nibbles 0..7) into an f16 pair:
//   nibbles (0, 4) -> (1024 + c0, 1024 + c4)
//   nibbles (1, 5) -> (1024 + 16 c1, 1024 + 16 c5)
// and the word shifted right by 8 gives nibbles (2, 6) and (3, 7) the same
// way.  The token operand carries q opposite the first kind and q / 16
// opposite the second (both exact in f16), so every product is an integer:
//   (1024 + c) q = 1024 q + c q,      (1024 + 16 c) q / 16 = 64 q + c q.
// The accumulator starts at -(1024 Q_even + 64 Q_odd) (Q_even / Q_odd: sums
// of q over the even / odd k of the group), so after the group's MMAs it holds
// exactly D = sum_k c q (every partial sum an integer below 2^20), and
//   I = sum_k q (c - z) = D - z qs
// exactly in fp32.  The k order inside the MMA is one permutation applied to
// both operands, so each thread's 16-byte weight loads (32 codes of rows r
// and r + 8) feed its A fragments directly.  Token fragments (f16 pairs) and
// the per-group offsets are built once per CTA in shared memory.
//
// Work split: persistent CTAs over 16-row tiles; an item is a tile and a pair
// of adjacent groups; the 8 warps of a CTA split a tile's pairs; each tile's
// group integers go to shared memory and one warp folds them in ascending
// group order while the others start the next tile (double-buffered).
// ---------------------------------------------------------------------------
namespace hm {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one weight word -> (c0, c4), (16 c1, 16 c5), (c2, c6), (16 c3, 16 c7), each + 1024
__device__ __forceinline__ void codes_f16(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t magic = 0x64006400u;
    p[0] = (w & 0x000F000Fu) | magic;
    p[1] = (w & 0x00F000F0u) | magic;
    const uint32_t t = w >> 8;
    p[2] = (t & 0x000F000Fu) | magic;
    p[3] = (t & 0x00F000F0u) | magic;
}

// one group of a 16-row tile: 8 MMAs over the thread's 4 words of rows r, r + 8
__device__ __forceinline__ void group_mma(float (&d)[4], const uint4 &wr0, const uint4 &wr1, const uint4 *bf) {
    const uint32_t w0[4] = {wr0.x, wr0.y, wr0.z, wr0.w}, w1[4] = {wr1.x, wr1.y, wr1.z, wr1.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 b = bf[u * 4];
        uint32_t a0[4], a1[4];
        codes_f16(w0[u], a0);
        codes_f16(w1[u], a1);
        mma_f16_16816(d, a0[0], a1[0], a0[1], a1[1], b.x, b.y);
        mma_f16_16816(d, a0[2], a1[2], a0[3], a1[3], b.z, b.w);
    }
}

__device__ __forceinline__ uint32_t f16_pair(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// signed 4-bit activation code i of a word, as a float
__device__ __forceinline__ float act_code(uint32_t w, int i) {
    return (float)((int32_t)(w << (28 - 4 * i)) >> 28);
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v >> 16))); }

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// shared memory: token fragments uint4 [MT + 1][G * 16 + 4] (padded per
// token; slot MT stays zero for the lanes of absent tokens), {offset, qs}
// float2 [G][MT], sx float [MT][G], I float [2][G][16][MT], scale words
// uint32 [2][G][16]
inline size_t smem_bytes(int MT, int K) {
    const size_t G = (size_t)K / kGroup;
    return (size_t)(MT + 1) * (G * 16 + 4) * 16 + (size_t)MT * G * 8 + (size_t)MT * G * 4 + 2 * G * 16 * MT * 4 +
           2 * G * 16 * 4;
}

// One item: a 16-row tile and a pair of adjacent groups (g0, g0 + 1), the
// thread's 16-byte pieces of rows r, r + 8 and their scale words.
struct Item {
    uint4 w00, w01, w10, w11;     // [row r / r + 8][group g0 / g0 + 1]
    uint32_t z00, z01, z10, z11;
};

// kPrefetch: items in flight per warp; kMinBlocks: CTAs per SM the register
// budget is sized for
template <int MT, int kPrefetch, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    w4a4_hmma_gemv_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ sx,
                          const int32_t *__restrict__ qs, const uint8_t *__restrict__ packed,
                          const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y, int ldy,
                          int32_t *__restrict__ dbg_I, const uint16_t *__restrict__ x, int ldx,
                          uint8_t *__restrict__ xq_out, float *__restrict__ sx_out, int32_t *__restrict__ qs_out,
                          int32_t *__restrict__ st) {
    static_assert(MT >= 1 && MT <= 8 && (MT == 1 || MT % 2 == 0), "one n8 block of tokens");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = K / kGroup;
    const int P = (G + 1) / 2;                                   // group pairs per row
    const size_t tstride = (size_t)G * 16 + 4;
    uint4 *bfr = reinterpret_cast<uint4 *>(smem_raw);
    float2 *oq = reinterpret_cast<float2 *>(bfr + (size_t)(MT + 1) * tstride);
    float *sxs = reinterpret_cast<float *>(oq + (size_t)MT * G);
    float *ibuf = sxs + (size_t)MT * G;
    uint32_t *sbuf = reinterpret_cast<uint32_t *>(ibuf + (size_t)2 * G * 16 * MT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qr = lane >> 2, qc = lane & 3;
    const int tok0 = blockIdx.y * MT;
    const int n_tiles = (N + 15) / 16;
    const size_t row_bytes = (size_t)K / 2;
    const int ngw = warp < P ? (P - warp + kWarps - 1) / kWarps : 0;   // this warp's pairs per tile
    const int my_tiles = (int)blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int n_items = ngw * my_tiles;
    // scale words of a pair in one 8-byte load when every pair is complete and aligned
    const bool z64 = (G % 2 == 0) && ((reinterpret_cast<uintptr_t>(sz) & 7) == 0);

    // producer cursor: tile step, pair index and the tile's row pointers
    // (rows past N read row 0; their results are never stored)
    struct Prod {
        int step, j;
        const uint8_t *p0, *p1;
        const uint32_t *z0, *z1;
    };
    auto set_tile = [&](Prod &c) {
        const int r0 = (blockIdx.x + c.step * gridDim.x) * 16 + qr, r1 = r0 + 8;
        const int s0 = r0 < N ? r0 : 0, s1 = r1 < N ? r1 : 0;
        c.p0 = packed + (size_t)s0 * row_bytes + qc * 16;
        c.p1 = packed + (size_t)s1 * row_bytes + qc * 16;
        c.z0 = sz + (size_t)s0 * G;
        c.z1 = sz + (size_t)s1 * G;
    };
    auto load_item = [&](const Prod &c, Item &x) {
        const int g0 = 2 * (warp + c.j * kWarps);
        const int d1 = g0 + 1 < G ? 1 : 0;                       // an odd last group pairs with itself
        const uint4 *a = reinterpret_cast<const uint4 *>(c.p0 + (size_t)g0 * 64);
        const uint4 *b = reinterpret_cast<const uint4 *>(c.p1 + (size_t)g0 * 64);
        x.w00 = ldg_stream(a);
        x.w01 = ldg_stream(a + d1 * 4);
        x.w10 = ldg_stream(b);
        x.w11 = ldg_stream(b + d1 * 4);
        if (z64) {
            const uint2 za = __ldg(reinterpret_cast<const uint2 *>(c.z0 + g0));
            const uint2 zb = __ldg(reinterpret_cast<const uint2 *>(c.z1 + g0));
            x.z00 = za.x;
            x.z01 = za.y;
            x.z10 = zb.x;
            x.z11 = zb.y;
        } else {
            x.z00 = __ldg(c.z0 + g0);
            x.z01 = __ldg(c.z0 + g0 + d1);
            x.z10 = __ldg(c.z1 + g0);
            x.z11 = __ldg(c.z1 + g0 + d1);
        }
    };
    auto advance_prod = [&](Prod &c) {
        if (++c.j == ngw) {
            c.j = 0;
            ++c.step;
            set_tile(c);
        }
    };

    pdl_launch_dependents();
    // immutable weights and scale words first
    Item ring[kPrefetch];
    Prod pc = {0, 0, nullptr, nullptr, nullptr, nullptr};
    set_tile(pc);
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p) {
        if (p < n_items) {
            load_item(pc, ring[p]);
            advance_prod(pc);
        }
    }
    pdl_wait();

    // token fragments, one thread per activation word (8 codes); the 16 words
    // of a group sit in 16 consecutive lanes, which reduce the group offset.
    // With x given, the words come from quantising x here (the a2 step, the
    // same routine as the quantiser; CTA column 0 also stores xq, sx, qs).
    const int wpr = K / 8;
    const bool fused = x != nullptr;
    bool bad = false;
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(xq);
    constexpr int kBatch = 4;                              // loads in flight per thread
    for (int base = 0; base < MT * wpr; base += kBatch * kThreads) {
        uint4 xv[kBatch];
        uint32_t wv[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = base + b * kThreads + threadIdx.x;
            const int t = i / wpr, wi = i - t * wpr;
            const bool live = i < MT * wpr && tok0 + t < M;
            if (fused)
                xv[b] = live ? *reinterpret_cast<const uint4 *>(x + (size_t)(tok0 + t) * ldx + (size_t)wi * 8)
                             : make_uint4(0u, 0u, 0u, 0u);
            else
                wv[b] = live ? xw[(size_t)(tok0 + t) * wpr + wi] : 0u;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = base + b * kThreads + threadIdx.x;
            const bool valid = i < MT * wpr;
            const int t = valid ? i / wpr : 0, wi = i - t * wpr;
            const bool live = valid && tok0 + t < M;
            uint32_t w = wv[b];
            if (fused) {
                float scale;
                int qsum;
                w = quant_group_halfwarp(xv[b], scale, qsum, bad);
                if (live) {
                    const int m = tok0 + t, g = wi >> 4;
                    if ((wi & 15) == 0) {
                        sxs[t * G + g] = scale;
                        oq[g * MT + t].y = (float)qsum;
                    }
                    if (blockIdx.x == 0) {
                        reinterpret_cast<uint32_t *>(xq_out + (size_t)m * (K / 2))[wi] = w;
                        if ((wi & 15) == 0) {
                            sx_out[(size_t)m * G + g] = scale;
                            qs_out[(size_t)m * G + g] = qsum;
                        }
                    }
                }
            }
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = act_code(w, e);
            float part = 1024.0f * ((q[0] + q[2]) + (q[4] + q[6])) + 64.0f * ((q[1] + q[3]) + (q[5] + q[7]));
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (valid) {
                const int g = wi >> 4, qcw = (wi >> 2) & 3, u = wi & 3;
                bfr[(size_t)t * tstride + (g * 4 + u) * 4 + qcw] =
                    make_uint4(f16_pair(q[0], q[4]), f16_pair(q[1] * 0.0625f, q[5] * 0.0625f), f16_pair(q[2], q[6]),
                               f16_pair(q[3] * 0.0625f, q[7] * 0.0625f));
                if ((wi & 15) == 0) oq[g * MT + t].x = part;
            }
        }
    }
    for (int i = threadIdx.x; i < (int)tstride; i += kThreads) bfr[(size_t)MT * tstride + i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < MT * G; i += kThreads) {
        const int t = i / G, g = i - t * G, m = tok0 + t;
        if (fused && m < M) continue;                    // set while quantising
        oq[g * MT + t].y = m < M ? (float)qs[(size_t)m * G + g] : 0.0f;
        sxs[i] = m < M ? sx[(size_t)m * G + g] : 0.0f;
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
    __syncthreads();

    // lanes of absent token columns read the zero slot
    const uint4 *brow = bfr + (size_t)(qr < MT ? qr : MT) * tstride + qc;
    // this lane's D columns are tokens 2 qc, 2 qc + 1 (clamped for the
    // offset loads; columns past MT are never stored)
    const int tq = MT == 1 ? 0 : (2 * qc < MT ? 2 * qc : 0);

    // end of tile `step`: every warp arrives once per tile; then one warp folds it
    auto tile_done = [&](int step) {
        __syncthreads();
        if (warp != (step & (kWarps - 1))) return;
        const int tile = blockIdx.x + step * gridDim.x;
        const float *ib = ibuf + (size_t)(step & 1) * G * 16 * MT;
        const uint32_t *sbb = sbuf + (size_t)(step & 1) * G * 16;
        for (int p = lane; p < 16 * MT; p += 32) {
            const int r = p / MT, t = p - (p / MT) * MT, n = tile * 16 + r, m = tok0 + t;
            if (n >= N || m >= M) continue;
            const float *ip = ib + (size_t)r * MT + t;
            const uint32_t *sp = sbb + r;
            const float *xp = sxs + (size_t)t * G;
            float acc = 0.0f;
#pragma unroll 4
            for (int g = 0; g < G; ++g)
                acc = __fmaf_rn(ip[(size_t)g * 16 * MT], __fmul_rn(xp[g], half_lo(sp[g * 16])), acc);
            y[(size_t)m * ldy + n] = float_to_bf16_bits(acc);
            if (dbg_I)
                for (int g = 0; g < G; ++g) dbg_I[((size_t)m * N + n) * G + g] = (int32_t)ip[(size_t)g * 16 * MT];
        }
    };

    // group g: D starts at minus the token offsets, so after the MMAs
    // D = sum c q and I = D - z qs (rows qr, qr + 8 x tokens 2 qc, 2 qc + 1)
    auto group = [&](const uint4 &wr0, const uint4 &wr1, uint32_t za, uint32_t zb, int g, float *ib,
                     uint32_t *sbb) {
        float d[4];
        float qs0, qs1;
        if (MT == 1) {
            const float2 o = oq[g];
            d[0] = d[1] = d[2] = d[3] = -o.x;
            qs0 = qs1 = o.y;
        } else {
            const float4 o = *reinterpret_cast<const float4 *>(oq + g * MT + tq);
            d[0] = d[2] = -o.x;
            d[1] = d[3] = -o.z;
            qs0 = o.y;
            qs1 = o.w;
        }
        group_mma(d, wr0, wr1, brow + (size_t)g * 16);
        const float zfa = half_hi(za), zfb = half_hi(zb);
        if (2 * qc < MT) {
            float *i0 = ib + ((size_t)g * 16 + qr) * MT + 2 * qc;
            float *i1 = i0 + 8 * MT;
            i0[0] = __fmaf_rn(-zfa, qs0, d[0]);
            i1[0] = __fmaf_rn(-zfb, qs0, d[2]);
            if (MT > 1) {
                i0[1] = __fmaf_rn(-zfa, qs1, d[1]);
                i1[1] = __fmaf_rn(-zfb, qs1, d[3]);
            }
        }
        if (qc == 0) {
            sbb[(size_t)g * 16 + qr] = za;
            sbb[(size_t)g * 16 + qr + 8] = zb;
        }
    };

    int cj = 0, cstep = 0;                                 // consumer cursor
    int cur = 0;                                           // tile step being produced
    for (int base = 0; base < n_items; base += kPrefetch) {
#pragma unroll
        for (int p = 0; p < kPrefetch; ++p) {
            const int it = base + p;
            if (it >= n_items) break;
            if (cstep != cur) {                            // this warp's first item of the next tile
                tile_done(cur);
                cur = cstep;
            }
            const int g0 = 2 * (warp + cj * kWarps);
            float *ib = ibuf + (size_t)(cur & 1) * G * 16 * MT;
            uint32_t *sbb = sbuf + (size_t)(cur & 1) * G * 16;
            const Item x = ring[p];
            if (it + kPrefetch < n_items) {
                load_item(pc, ring[p]);
                advance_prod(pc);
            }
            group(x.w00, x.w10, x.z00, x.z10, g0, ib, sbb);
            if (g0 + 1 < G) group(x.w01, x.w11, x.z01, x.z11, g0 + 1, ib, sbb);
            if (++cj == ngw) {
                cj = 0;
                ++cstep;
            }
        }
    }
    // the last tile with items, then the remaining ones (warps without pairs)
    for (; cur < my_tiles; ++cur) tile_done(cur);
}

// Quantised activations as input (x == nullptr), or bf16 x quantised in the
// kernel with xq, sx, qs stored as outputs.
struct Act {
    const uint8_t *xq;
    const float *sx;
    const int32_t *qs;
    const uint16_t *x;
    int ldx;
    uint8_t *xq_out;
    float *sx_out;
    int32_t *qs_out;
};

template <int MT, int PF = 1, int MINB = 2>
int launch(const Act &a, const uint8_t *packed, const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy,
           int32_t *dbg_I, int32_t *dev_status, cudaStream_t st, int ctas_per_sm = MINB) {
    const size_t smem = smem_bytes(MT, K);
    auto kern = w4a4_hmma_gemv_kernel<MT, PF, MINB>;
    int rc = smem_limit_once(reinterpret_cast<const void *>(kern), 200 * 1024);
    if (rc) return rc;
    const int n_tiles = (N + 15) / 16, token_tiles = (M + MT - 1) / MT;
    const int per_col = std::max(1, ctas_per_sm * sm_count() / token_tiles);
    dim3 grid((unsigned)std::min(n_tiles, per_col), (unsigned)token_tiles);
    return launch_pdl("qspec_linear_w4a4", kern, grid, dim3(kThreads), smem, st, a.xq, a.sx, a.qs, packed, sz, M, N,
                      K, y, ldy, dbg_I, a.x, a.ldx, a.xq_out, a.sx_out, a.qs_out, dev_status);
}

// tokens per CTA of the warp-MMA path: up to 8 (one MMA column block),
// halved while two CTAs would not fit on an SM
int tokens_per_cta(int M, int K) {
    constexpr size_t kTwoPerSm = 112 * 1024;
    int mt = M == 1 ? 1 : M == 2 ? 2 : M <= 4 ? 4 : 8;
    while (mt > 1 && smem_bytes(mt, K) > kTwoPerSm) mt /= 2;
    return mt;
}

// up to 32 tokens go to the tensor-core kernel (all tokens of a 128-row tile
// in one CTA) when the warp-MMA path would read the weights more than 12
// times (large K leaves room for few tokens per warp-MMA CTA), and 17..32
// tokens on the larger layers (N >= 6144), where it measured 1.2-2.5x faster
// than the warp-MMA kernel's several token tiles (LM head at 32 tokens: 216
// vs 547 us) even with its separate quantiser launch; and from 9 tokens on
// every layer, where its 16-token tiles with the groups split over 2- or
// 4-CTA clusters beat two warp-MMA token tiles (16 tokens: 6144 x 4096 30 ->
// 27 us, 4096 x 4096 25 -> 18 us; 12 tokens, 4096 x 14336: 97 -> 35 us)
bool use_tc(int M, int N, int K) {
    const int mt = tokens_per_cta(M, K);
    return M >= 9 || (M + mt - 1) / mt > 12 || (M > 16 && N >= 6144);
}

// warp-MMA path for M <= 32: QSPEC_ERR_SHAPE when the shape does not fit
int launch_small(const Act &a, const uint8_t *packed, const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy,
                 int32_t *dbg_I, int32_t *dev_status, cudaStream_t st) {
    constexpr size_t kMaxSmem = 200 * 1024;
    const int mt = tokens_per_cta(M, K);
    if (smem_bytes(mt, K) > kMaxSmem) return QSPEC_ERR_SHAPE;
    switch (mt) {
        case 1: return launch<1>(a, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, st);
        case 2: return launch<2>(a, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, st);
        case 4: return launch<4>(a, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, st);
        default: return launch<8>(a, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, st);
    }
}

// the tensor-memory GEMV takes 3..16 tokens when every SM gets a 128-row tile
// (9..16 tokens with fewer than 4 tiles per SM: the tensor-core kernel's
// 16-token tiles measured faster, 28672 x 4096 at 16 tokens 35.2 -> 29.7 us;
// the LM head stays here, 99.6 vs 107.8 us)
bool use_gemv_tc(int M, int N) {
    const int tiles = (N + 127) / 128;
    return M >= 3 && M <= 16 && tiles >= sm_count() && (M <= 8 || tiles >= 4 * sm_count());
}

}  // namespace hm

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
    if (M > 32) return launch_w4a4_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st, kWaitLimit, 0);
    if (M == 1) {
        rc = launch_w4a4_dp4a(xq, sx, qs, nullptr, nullptr, nullptr, nullptr, packed, sz, N, K, y_bf16, dbg_I,
                              dev_status, st);
        if (rc != QSPEC_ERR_SHAPE) return rc;
    }
    // 3..16 tokens and at least one 128-row tile per SM: weights through TMA
    // and TMEM, MMAs async (at 1-2 tokens the warp-MMA kernel below is faster)
    if (hm::use_gemv_tc(M, N)) {
        rc = launch_w4a4_gemv_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st, kWaitLimit, 0);
        if (rc != QSPEC_ERR_SHAPE) return rc;
    }
    if (hm::use_tc(M, N, K)) return launch_w4a4_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st, kWaitLimit, 0);
    const hm::Act act = {xq, sx, qs, nullptr, 0, nullptr, nullptr, nullptr};
    return hm::launch_small(act, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st);
}

extern "C" int qspec_linear_w4a4_bf16(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz,
                                      int M, int N, int K, uint16_t *y_bf16, int ldy, uint8_t *xq, float *sx,
                                      int32_t *qs, int32_t *dbg_I, int32_t *dev_status, qspec_stream_t stream) {
    if (!x_bf16 || !packed || !sz || !y_bf16 || !xq || !sx || !qs) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < kGroup || K % kGroup || ldx < K || ldy < N) return QSPEC_ERR_SHAPE;
    if (!aligned(x_bf16, 16) || ldx % 8 || !aligned(xq, 16) || !aligned(sx, 4) || !aligned(qs, 4) ||
        !aligned(packed, 16) || !aligned(sz, 4) || !aligned(y_bf16, 2) || (dbg_I && !aligned(dbg_I, 4)))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    if (M == 1) {
        rc = launch_w4a4_dp4a(nullptr, nullptr, nullptr, x_bf16, xq, sx, qs, packed, sz, N, K, y_bf16, dbg_I,
                              dev_status, st);
        if (rc != QSPEC_ERR_SHAPE) return rc;
    }
    if (M <= 32 && !hm::use_gemv_tc(M, N) && !hm::use_tc(M, N, K)) {
        const hm::Act act = {xq, sx, qs, x_bf16, ldx, xq, sx, qs};
        rc = hm::launch_small(act, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, st);
        if (rc != QSPEC_ERR_SHAPE) return rc;
    }
    // the other paths: the quantiser, then the linear on its outputs
    rc = qspec_quant_act_int4(x_bf16, M, K, ldx, xq, sx, qs, dev_status, stream);
    if (rc) return rc;
    return qspec_linear_w4a4(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, dbg_I, dev_status, stream);
}
