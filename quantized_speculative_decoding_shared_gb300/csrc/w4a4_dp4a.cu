// w4a4_dp4a.cu -- a3 for a single token (M = 1, the draft decode shape):
// the W4A4 linear on the integer byte dot-product unit.
//
// QSPEC summary page, background terms: W4A4 runs a low-precision kernel on
// 4-bit weights and 4-bit activations with no dequantisation, accumulating in
// INT32 before scaling to a 16-bit result.  Same bit-exact definition as the
// other W4A4 paths:
//   I[n][g] = sum_{k in g} q[k] (W[n][k] - z[n][g])
//   acc = 0; for g ascending: acc = fmaf((float) I, sx[g] * s[n][g], acc)
//   y[n] = bf16_rn(acc)
//
// At one token the f16 warp MMA wastes seven of its eight columns and the
// kernel is bound by instruction issue, not by HBM.  Here a weight word (codes
// c0..c7, low nibble = even k) feeds two 4-way byte dot products with no
// unpacking beyond two masks:
//   w & 0x0F0F0F0F = bytes (c0, c2, c4, c6)         times (16 q0, 16 q2, ...)
//   w & 0xF0F0F0F0 = bytes (16 c1, 16 c3, ...)       times (q1, q3, ...)
// so dp4a(lo, E) + dp4a(hi, O) = 16 sum_k c q exactly (unsigned weight bytes,
// signed activation bytes: 16 q is in [-128, 112] even for the code -8).  The
// activation bytes E, O are built once per CTA in shared memory.
//
// Work split: a unit is 512 contiguous bytes of one row (1024 codes = eight
// groups), one 16-byte piece per lane.  Each CTA owns a contiguous, balanced
// range of rows, walked in chunks of RC rows; in a chunk the warps take
// units round-robin (at most kUnits each).  Each thread streams its pieces
// into its own slots of a shared-memory ring with asynchronous copies, two
// chunks ahead of the one being reduced.  After the four
// lanes of a group combine their sums, each group's exact I and sx * s go to
// shared memory, and one thread per row folds them in ascending group order
// (overlapping the next chunk).  Every CTA builds the activation bytes of
// the whole vector, quantising x itself when given.
#include <algorithm>
#include <type_traits>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {

namespace dq {

constexpr int kSegGroups = 8;       // groups per unit (512 bytes of a row)
constexpr int kUnits = 8;           // units per warp and chunk

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 16 bytes global -> shared, asynchronous; src_bytes 0 writes zeros and reads nothing
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc), "r"(src_bytes), "l"(policy)
                 : "memory");
}

// Block-wide barrier that warps may reach from different places in the code
// (the non-aligned form): unit warps, fold warps and the two copies of the
// chunk loop each meet it once per chunk.
__device__ __forceinline__ void cta_barrier() { asm volatile("barrier.sync 0;\n" ::: "memory"); }

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v >> 16))); }

// activation word (codes q0..q7, two's complement nibbles) -> the byte
// operands E' = (16 q0 - q1, 16 q2 - q3, ...) (mod 256) and O = (q1, q3, q5,
// q7); `m8` is set when an even code is -8 (then 16 q0 - q1 may not fit a
// signed byte)
__device__ __forceinline__ void act_bytes(uint32_t nib, uint32_t &ep, uint32_t &o, bool &m8) {
    const uint32_t lo = nib & 0x0F0F0F0Fu;
    o = __vsub4(((nib >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u, 0x08080808u);
    ep = __vsub4(lo << 4, o);
    m8 |= __vcmpeq4(lo, 0x08080808u) != 0u;
}

// 16 x the dot product of one 16-byte weight piece with its activation
// bytes, when no even code is -8:
//   dp4a(w, O) + dp4a(w & 0x0F0F0F0F, E')
//     = sum (c_e + 16 c_o) q_o + c_e (16 q_e - q_o) = 16 sum (c_e q_e + c_o q_o)
__device__ __forceinline__ int piece_dot(const uint4 &w, const uint4 &ep, const uint4 &o) {
    int p = 0;
    p = dp4a_us(w.x, o.x, p);
    p = dp4a_us(w.x & 0x0F0F0F0Fu, ep.x, p);
    p = dp4a_us(w.y, o.y, p);
    p = dp4a_us(w.y & 0x0F0F0F0Fu, ep.y, p);
    p = dp4a_us(w.z, o.z, p);
    p = dp4a_us(w.z & 0x0F0F0F0Fu, ep.z, p);
    p = dp4a_us(w.w, o.w, p);
    p = dp4a_us(w.w & 0x0F0F0F0Fu, ep.w, p);
    return p;
}

// The same for any codes: E' + O = 16 q_e (mod 256, in [-128, 112]) against
// the low nibbles, O against the high nibbles (16 c_o).
__device__ __forceinline__ int piece_dot_any(const uint4 &w, const uint4 &ep, const uint4 &o) {
    int p = 0;
    p = dp4a_us(w.x & 0x0F0F0F0Fu, __vadd4(ep.x, o.x), p);
    p = dp4a_us(w.x & 0xF0F0F0F0u, o.x, p);
    p = dp4a_us(w.y & 0x0F0F0F0Fu, __vadd4(ep.y, o.y), p);
    p = dp4a_us(w.y & 0xF0F0F0F0u, o.y, p);
    p = dp4a_us(w.z & 0x0F0F0F0Fu, __vadd4(ep.z, o.z), p);
    p = dp4a_us(w.z & 0xF0F0F0F0u, o.z, p);
    p = dp4a_us(w.w & 0x0F0F0F0Fu, __vadd4(ep.w, o.w), p);
    p = dp4a_us(w.w & 0xF0F0F0F0u, o.w, p);
    return p;
}

// Shared memory: the weight ring uint4 [P][kUnits][unit threads] (each
// thread's own pieces of P chunks), activation bytes uint4 [S][2][32] (E', O
// of each lane's four words of a unit), (I, sx s) float2 [2][RC][pstride >
// G], sx float [G], qs float [G].
inline size_t smem_bytes(int K, int RC, int unit_threads, int P) {
    const size_t G = (size_t)K / kGroup, S = (G + kSegGroups - 1) / kSegGroups;
    const size_t pstride = (G + 13) / 16 * 16 + 2;
    return (size_t)P * kUnits * unit_threads * 16 + S * 64 * 16 + G * 8 + 2 * (size_t)RC * pstride * 8;
}

// blockDim.x / 32 <= kMaxWarps warps, the first nw of which reduce units
// (the rest, if any, fold the groups); RC: rows per chunk (RC * S <= nw *
// kUnits).  x == nullptr: xq, sx, qs are the quantised activations; else x
// (bf16) is quantised here and CTA 0 stores xq_out, sx_out, qs_out.
// kFixed: S divides nw, so every unit of a warp has the same segment
// (warp % S) and the next unit's row is nw / S further; the warp keeps that
// segment's activation bytes in registers.  kP: chunks of weights in the
// shared-memory ring (kP - 1 in flight while one is reduced).
template <int kMaxWarps, bool kFixed, int kP>
__global__ void __launch_bounds__(kMaxWarps * 32, 16 / kMaxWarps)
    w4a4_dp4a_gemv_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ sx,
                          const int32_t *__restrict__ qs, const uint8_t *__restrict__ packed,
                          const uint32_t *__restrict__ sz, int N, int K, int nw, int RC, uint16_t *__restrict__ y,
                          int32_t *__restrict__ dbg_I, const uint16_t *__restrict__ x, uint8_t *__restrict__ xq_out,
                          float *__restrict__ sx_out, int32_t *__restrict__ qs_out, int32_t *__restrict__ st) {
    const int kThreads = (int)blockDim.x, kCThreads = nw * 32;   // all threads, unit threads
    const bool fold_warps = kThreads > kCThreads;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = K / kGroup;
    const int S = (G + kSegGroups - 1) / kSegGroups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 *ring = reinterpret_cast<uint4 *>(smem_raw);
    uint4 *act = ring + (size_t)kP * kUnits * kCThreads;
    // (I, sx s) row stride: 16-byte aligned rows, consecutive rows 16 bytes
    // apart modulo 128 (conflict-free 16-byte reads by consecutive threads)
    const int pstride = (G + 13) / 16 * 16 + 2;
    float2 *pairs = reinterpret_cast<float2 *>(act + (size_t)S * 64);
    float *sxs = reinterpret_cast<float *>(pairs + (size_t)2 * RC * pstride);
    float *qss = sxs + G;
    const size_t row_bytes = (size_t)K / 2;

    const int r_begin = (int)(((long long)blockIdx.x * N) / gridDim.x);
    const int r_end = (int)(((long long)(blockIdx.x + 1) * N) / gridDim.x);
    const int n_chunks = (r_end - r_begin + RC - 1) / RC;

    // unit j of this warp in every chunk: u = warp + j * nw, row u / S,
    // segment u % S (both below 128, kept as bytes); lanes whose group is
    // past G load nothing
    uint32_t rows_of[kUnits / 4] = {}, segs[kUnits / 4] = {};
    uint32_t lane_ok = 0, off0 = 0, dj = 0;
    if constexpr (kFixed) {
        off0 = (uint32_t)(warp / S) * (uint32_t)row_bytes + (uint32_t)(warp % S) * 512u;
        dj = (uint32_t)(nw / S) * (uint32_t)row_bytes;
        lane_ok = ((warp % S) * kSegGroups + (lane >> 2) < G) ? 0xFFu : 0u;
    } else {
#pragma unroll
        for (int j = 0; j < kUnits; ++j) {
            const int u = warp + j * nw, rl = u / S, sg = u - rl * S;
            rows_of[j / 4] |= (uint32_t)(rl & 0xFF) << (8 * (j % 4));
            segs[j / 4] |= (uint32_t)sg << (8 * (j % 4));
            if (sg * kSegGroups + (lane >> 2) < G) lane_ok |= 1u << j;
        }
    }
    const uint8_t *lane_base = packed + (size_t)lane * 16;
    // after the reduction of batch b, lane 4 g' + i holds unit 4 b + i, group
    // g' of its segment: the same unit, row slot and group in every chunk
    int eu[2], erl[2], eg[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        eu[b] = warp + (4 * b + (lane & 3)) * nw;
        erl[b] = eu[b] / S;
        eg[b] = (eu[b] - erl[b] * S) * kSegGroups + (lane >> 2);
        if (eg[b] >= G) eu[b] = 1 << 30;                  // never valid
    }

    // weights are read once: first out of L2
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(policy));
    auto chunk_rows = [&](int c) { return min(RC, r_end - (r_begin + c * RC)); };
    // chunk c's weight pieces into ring stage c % kP (each thread its own),
    // one commit group per call, empty past the last chunk
    auto issue = [&](int c) {
        if (c < n_chunks) {
            const int row0 = r_begin + c * RC, n_units = chunk_rows(c) * S;
            const uint8_t *base = lane_base + (size_t)row0 * row_bytes;
            uint4 *dst = ring + (size_t)(c % kP) * kUnits * kCThreads + threadIdx.x;
#pragma unroll
            for (int j = 0; j < kUnits; ++j) {
                const uint32_t off = kFixed ? off0 + (uint32_t)j * dj
                                            : ((rows_of[j / 4] >> (8 * (j % 4))) & 0xFFu) * (uint32_t)row_bytes +
                                                  ((segs[j / 4] >> (8 * (j % 4))) & 0xFFu) * 512u;
                const bool ok = warp + j * nw < n_units && (lane_ok >> j & 1u);
                cp_async16(dst + (size_t)j * kCThreads, ok ? base + off : packed, ok ? 16u : 0u, policy);
            }
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };
    auto load_sz = [&](int c, uint32_t (&zw)[2]) {
        const int row0 = r_begin + c * RC, n_units = chunk_rows(c) * S;
#pragma unroll
        for (int b = 0; b < 2; ++b)
            zw[b] = eu[b] < n_units ? __ldg(sz + (size_t)(row0 + erl[b]) * G + eg[b]) : 0u;
    };

    pdl_launch_dependents();
    // immutable weights before the wait: the first kP - 1 chunks
    const bool unit_warp = warp < nw;
    uint32_t za[2] = {0u, 0u}, zb[2] = {0u, 0u};
    if (unit_warp) {
#pragma unroll
        for (int c = 0; c < kP - 1; ++c) issue(c);
        if (n_chunks > 0) load_sz(0, za);
    }
    pdl_wait();

    // Activation bytes, and sx, qs of the epilogue groups.
    //  kFixed, with the quantised activations given or one unit warp per
    //   segment (nw == S): a warp's units all lie in segment warp % S, and
    //   lane l's 16-byte pieces are codes 32 l .. 32 l + 31 of the segment,
    //   a quarter of group l / 4: each unit warp builds (quantising x when
    //   given, four lanes per group) exactly the bytes its lanes need, in
    //   registers, with no block-wide step; its epilogue groups are its
    //   lanes' own groups.
    //  Otherwise (where quantising that way would repeat work): the CTA
    //   builds the whole vector in shared memory, each group once.
    bool bad = false, m8 = false, any_m8 = false;
    uint4 fe = make_uint4(0u, 0u, 0u, 0u), fo = fe;
    float esx[2] = {0.0f, 0.0f}, eqs[2] = {0.0f, 0.0f};
    if (kFixed && (x == nullptr || nw == S)) {
        if (unit_warp) {
            const int sg = warp % S, g = sg * kSegGroups + (lane >> 2);
            const bool live = g < G;
            uint32_t nib[4] = {0u, 0u, 0u, 0u};
            float scale = 0.0f, qsf = 0.0f;
            if (x == nullptr) {
                if (live) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(xq + (size_t)sg * 512 + lane * 16);
                    nib[0] = w.x;
                    nib[1] = w.y;
                    nib[2] = w.z;
                    nib[3] = w.w;
                    scale = sx[g];
                    qsf = (float)qs[g];
                }
            } else {
                uint4 v[4];
                const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)sg * 1024 + lane * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = live ? src[i] : make_uint4(0u, 0u, 0u, 0u);
                int qsum;
                quant_group<4>(v, scale, qsum, bad, nib);
                qsf = (float)qsum;
                if (blockIdx.x == 0 && warp < S && live) {
                    *reinterpret_cast<uint4 *>(xq_out + (size_t)sg * 512 + lane * 16) =
                        make_uint4(nib[0], nib[1], nib[2], nib[3]);
                    if ((lane & 3) == 0) {
                        sx_out[g] = scale;
                        qs_out[g] = qsum;
                    }
                }
            }
            act_bytes(nib[0], fe.x, fo.x, m8);
            act_bytes(nib[1], fe.y, fo.y, m8);
            act_bytes(nib[2], fe.z, fo.z, m8);
            act_bytes(nib[3], fe.w, fo.w, m8);
            any_m8 = __any_sync(0xffffffffu, m8);
            esx[0] = esx[1] = scale;
            eqs[0] = eqs[1] = qsf;
        }
        if (bad) flag(st, QSPEC_ERR_NONFINITE);
    } else {
        const int words = K / 8;
        auto put_word = [&](int wi, uint32_t nib) {
            uint32_t ep, o;
            act_bytes(nib, ep, o, m8);
            uint32_t *a = reinterpret_cast<uint32_t *>(act + (size_t)(wi >> 7) * 64 + ((wi >> 2) & 31));
            a[wi & 3] = ep;
            a[128 + (wi & 3)] = o;
        };
        if (x == nullptr) {
            const uint32_t *xw = reinterpret_cast<const uint32_t *>(xq);
            constexpr int kB = 4;
            for (int w0 = threadIdx.x; w0 < S * 128; w0 += kB * kThreads) {
                uint32_t xw4[kB];
#pragma unroll
                for (int i = 0; i < kB; ++i) xw4[i] = w0 + i * kThreads < words ? xw[w0 + i * kThreads] : 0u;
#pragma unroll
                for (int i = 0; i < kB; ++i)
                    if (w0 + i * kThreads < S * 128) put_word(w0 + i * kThreads, xw4[i]);
            }
            for (int g = threadIdx.x; g < G; g += kThreads) {
                sxs[g] = sx[g];
                qss[g] = (float)qs[g];
            }
        } else {
            // eight lanes per group, 16 elements each (two 16-byte words); CTA 0
            // also stores xq, sx, qs
            const int sub = lane >> 3, l8 = lane & 7;
            const int kPer = kThreads / 8;                    // groups per pass: 4 per warp
            for (int g0 = 4 * warp; g0 < G; g0 += 2 * kPer) {
                uint4 v[2][2];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int g = g0 + p * kPer + sub;
                    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)g * kGroup) + 2 * l8;
                    v[p][0] = g < G ? src[0] : make_uint4(0u, 0u, 0u, 0u);
                    v[p][1] = g < G ? src[1] : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int g = g0 + p * kPer + sub;
                    if (g0 + p * kPer >= G) break;            // warp-uniform
                    float scale;
                    int qsum;
                    uint32_t nib[2];
                    quant_group<2>(v[p], scale, qsum, bad, nib);
                    if (g < G) {
                        const int wi = g * 16 + 2 * l8;
                        put_word(wi, nib[0]);
                        put_word(wi + 1, nib[1]);
                        if (l8 == 0) {
                            sxs[g] = scale;
                            qss[g] = (float)qsum;
                        }
                        if (blockIdx.x == 0) {
                            *reinterpret_cast<uint2 *>(xq_out + (size_t)wi * 4) = make_uint2(nib[0], nib[1]);
                            if (l8 == 0) {
                                sx_out[g] = scale;
                                qs_out[g] = qsum;
                            }
                        }
                    }
                }
            }
            // words of a partial last unit: zero (their weights load as zeros too)
            for (int wi = words + threadIdx.x; wi < S * 128; wi += kThreads) put_word(wi, 0u);
        }
        if (bad) flag(st, QSPEC_ERR_NONFINITE);
        any_m8 = __syncthreads_or(m8);
        if (kFixed && unit_warp) {
            fe = act[(warp % S) * 64 + lane];
            fo = act[(warp % S) * 64 + 32 + lane];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int g = eg[b] < G ? eg[b] : 0;
            esx[b] = sxs[g];
            eqs[b] = qss[g];
        }
    }
    // this lane's pair slots
    int pidx[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) pidx[b] = erl[b] * pstride + eg[b];

    // one thread per row folds the groups of chunk c in ascending order
    // (the fold warps' threads when there are any, else every thread)
    // (unit threads start past the last row when fold warps exist)
    const int f0 = !fold_warps ? (int)threadIdx.x : unit_warp ? RC : (int)threadIdx.x - kCThreads;
    const int fstep = fold_warps ? kThreads - kCThreads : kThreads;
    auto fold = [&](int c) {
        const int row0 = r_begin + c * RC, rows = chunk_rows(c);
        const float2 *pb = pairs + (size_t)(c & 1) * RC * pstride;
        for (int t = f0; t < rows; t += fstep) {
            const float4 *pp = reinterpret_cast<const float4 *>(pb + (size_t)t * pstride);
            float acc = 0.0f;
#pragma unroll 8
            for (int h = 0; h < G / 2; ++h) {
                const float4 v = pp[h];
                acc = __fmaf_rn(v.x, v.y, acc);
                acc = __fmaf_rn(v.z, v.w, acc);
            }
            if (G & 1) {
                const float4 v = pp[G / 2];
                acc = __fmaf_rn(v.x, v.y, acc);
            }
            y[row0 + t] = float_to_bf16_bits(acc);
        }
    };
    // one chunk: chunk c + kP - 1 into the stage chunk c - 1 left, the next
    // chunk's scale words, the previous chunk's fold, then (once chunk c's
    // pieces have landed) the dot products and the group epilogue
    // (two copies of the loop: codes -8 present or not, decided once)
    auto step = [&](auto any_tag, int c, uint32_t (&zc)[2], uint32_t (&zn)[2]) {
        constexpr bool kAny = decltype(any_tag)::value;
        if (!unit_warp) {
            if (c > 0) fold(c - 1);
            cta_barrier();
            return;
        }
        issue(c + kP - 1);
        if (c + 1 < n_chunks) load_sz(c + 1, zn);
        if (c > 0 && !fold_warps) fold(c - 1);
        asm volatile("cp.async.wait_group %0;\n" ::"n"(kP - 1) : "memory");
        const int row0 = r_begin + c * RC, n_units = chunk_rows(c) * S;
        float2 *pb = pairs + (size_t)(c & 1) * RC * pstride;
        const uint4 *cur = ring + (size_t)(c % kP) * kUnits * kCThreads + threadIdx.x;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            int part[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * b + i;
                uint4 e = fe, o = fo;
                if constexpr (!kFixed) {
                    const uint32_t a = ((segs[b] >> (8 * i)) & 0xFFu) * 64u + (uint32_t)lane;
                    e = act[a];
                    o = act[a + 32];
                }
                const uint4 w = cur[(size_t)j * kCThreads];
                if constexpr (kAny)
                    part[i] = piece_dot_any(w, e, o);
                else
                    part[i] = piece_dot(w, e, o);
            }
            // quad transpose-reduce: lane 4 g' + i ends with unit 4 b + i
            const int qi = lane & 3;
            const bool odd = qi & 1, upper = qi & 2;
            int k0 = odd ? part[1] : part[0], k1 = odd ? part[3] : part[2];
            const int s0 = odd ? part[0] : part[1], s1 = odd ? part[2] : part[3];
            k0 += __shfl_xor_sync(0xffffffffu, s0, 1);
            k1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            int d16 = upper ? k1 : k0;
            d16 += __shfl_xor_sync(0xffffffffu, upper ? k0 : k1, 2);
            if (eu[b] < n_units) {
                const float I = __fmaf_rn(-half_hi(zc[b]), eqs[b], (float)(d16 >> 4));
                pb[pidx[b]] = make_float2(I, __fmul_rn(esx[b], half_lo(zc[b])));
                if (dbg_I) dbg_I[(size_t)(row0 + erl[b]) * G + eg[b]] = (int32_t)I;
            }
        }
        cta_barrier();
    };
    auto run = [&](auto any_tag) {
        for (int c = 0; c < n_chunks; c += 2) {
            step(any_tag, c, za, zb);
            if (c + 1 < n_chunks) step(any_tag, c + 1, zb, za);
        }
    };
    if (any_m8)
        run(std::true_type{});
    else
        run(std::false_type{});
    if (n_chunks > 0) fold(n_chunks - 1);
    asm volatile("cp.async.wait_all;\n" ::: "memory");    // the empty tail groups
}

}  // namespace dq

}  // namespace

// One token: QSPEC_ERR_SHAPE before any launch when K is too long for a chunk
// of one row (more than 128 units of 1024 codes).
int launch_w4a4_dp4a(const uint8_t *xq, const float *sx, const int32_t *qs, const uint16_t *x, uint8_t *xq_out,
                     float *sx_out, int32_t *qs_out, const uint8_t *packed, const uint32_t *sz, int N, int K,
                     uint16_t *y, int32_t *dbg_I, int32_t *dev_status, cudaStream_t stream) {
    const int G = K / kGroup, S = (G + dq::kSegGroups - 1) / dq::kSegGroups;
    // up to 8 units per row: two 8-warp CTAs per SM; longer rows: one 16-warp
    // CTA.  When S <= warps, the unit warps are the largest multiple of S
    // (each warp's segment fixed) and the others fold the groups.
    const int max_w = S > 8 ? 16 : 8, per_sm = S > 8 ? 1 : 2;
    const bool fixed = S <= max_w;
    const int warps = fixed ? (max_w / S) * S : max_w;
    if (S > warps * dq::kUnits) return QSPEC_ERR_SHAPE;
    const int ctas = std::min(sm_count() * per_sm, N);
    const int rows_per_cta = (N + ctas - 1) / ctas;
    const int RC = std::min(warps * dq::kUnits / S, rows_per_cta);
    // a ring of 3 chunks when it fits (two CTAs per SM: half the SM each);
    // very long rows: 2, or 1 (no prefetch)
    const size_t budget = per_sm == 2 ? 112 * 1024 : 227 * 1024;
    int P = 3;
    while (P > 1 && dq::smem_bytes(K, RC, warps * 32, P) > budget) --P;
    const size_t smem = dq::smem_bytes(K, RC, warps * 32, P);
    if (smem > budget || (P < 2 && (max_w == 8 || fixed))) return QSPEC_ERR_SHAPE;
    void (*kern)(const uint8_t *, const float *, const int32_t *, const uint8_t *, const uint32_t *, int, int, int,
                 int, uint16_t *, int32_t *, const uint16_t *, uint8_t *, float *, int32_t *, int32_t *);
    if (max_w == 8)
        kern = P == 3 ? dq::w4a4_dp4a_gemv_kernel<8, true, 3> : dq::w4a4_dp4a_gemv_kernel<8, true, 2>;
    else if (fixed)
        kern = P == 3 ? dq::w4a4_dp4a_gemv_kernel<16, true, 3> : dq::w4a4_dp4a_gemv_kernel<16, true, 2>;
    else
        kern = P == 3 ? dq::w4a4_dp4a_gemv_kernel<16, false, 3>
               : P == 2 ? dq::w4a4_dp4a_gemv_kernel<16, false, 2>
                        : dq::w4a4_dp4a_gemv_kernel<16, false, 1>;
    int rc = smem_limit_once(reinterpret_cast<const void *>(kern), (int)smem, true);
    if (rc) return rc;
    return launch_pdl("qspec_linear_w4a4", kern, dim3((unsigned)ctas), dim3(max_w * 32), smem, stream, xq, sx, qs,
                      packed, sz, N, K, warps, RC, y, dbg_I, x, xq_out, sx_out, qs_out, dev_status);
}

}  // namespace qspec
