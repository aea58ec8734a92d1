// w4a4_gemv_tc.cu -- a3, W4A4 linear for decode-sized M (draft passes) on the
// Blackwell tensor cores, with the weight operand staged in tensor memory.
//
// QSPEC summary page, background terms: 4-bit weights times 4-bit
// activations, products accumulated exactly, then scaled to 16 bits; "QSPEC
// structure": the draft pass reads the same packed weights as the verify
// pass.  Bit-exact definition (shared with the other W4A4 kernels and the CPU
// oracle):
//   I[m][n][g] = sum_{k in g} q (W - z) ; acc = fmaf((float) I, sx * s, acc)
//   for g ascending from acc = 0 ; y = bf16_rn(acc).
//
// At decode M the linear streams the packed weights once; the kernel keeps
// the memory system busy with bulk tensor copies and spends few instructions
// per weight byte:
//   - warp 12 (one lane) streams 128-row x 128-byte boxes (a pair of groups
//     of a row tile) into a ring of shared-memory stages with TMA (128-byte
//     swizzle; rows past N arrive as zeros);
//   - warps 0-7 turn a stage into the MMA's A operand in tensor memory: one
//     E4M3 byte holding b in 0..15 is exactly b * 2^-9 (subnormal for b < 8,
//     exponent 1 above), so lo = w & 0x0F0F0F0F and hi = (w >> 4) & 0x0F0F0F0F
//     give one byte per code, written with tcgen05.st (warp w writes TMEM
//     lanes 32 (w % 4) + 16 (w / 4) .. + 15 = rows of the tile);
//   - warp 13 (one lane) runs per group 4 MMAs kind::f8f6f4 (M = 128, N = 16,
//     K = 32): A from TMEM, B = the tokens' q as E4M3 q * 2^-9 in shared
//     memory (token rows 0..7; rows 8..15 read the same rows again through a
//     zero row-group stride and are ignored); D = sum c q * 2^-18 exactly;
//   - warps 8-11 own the tile's rows for the epilogue (thread = TMEM lane =
//     output row): I = D * 2^18 - z qs exactly in fp32, folded into the row's
//     accumulators in group order, so no cross-thread reduction exists.
// Group pairs cycle through kPSlots TMEM slots (A 64 columns + D 32 columns
// each); one barrier round per pair.
// Every wait is bounded (the limit is a kernel argument; a test can also
// make the MMA issuer wait on a barrier nothing arrives at).  After a timeout
// (QSPEC_ERR_TIMEOUT) every role leaves its loop -- the producer and the MMA
// issuer issue nothing more -- the copies in flight and the MMAs issued are
// drained with bounded waits, and the kernel ends.  Should even the drain run
// out, the tensor memory is freed all the same: the next kernel on the SM
// would otherwise wait for it without a bound.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

namespace tg {

constexpr int kConvWarps = 8;              // two per TMEM lane quadrant, 16 rows each
constexpr int kEpiWarps = 4;               // one per quadrant, 32 rows each
constexpr int kProducerWarp = kConvWarps + kEpiWarps;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kPSlots = 4;                 // group pairs in flight through TMEM
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 0;              // A of pair slot s: columns 64 s .. 64 s + 63 (2 x 128 codes per lane)
constexpr uint32_t kDcol = 256;            // D of pair slot s: columns 256 + 32 s + 16 gi .. + 15
constexpr int kStageBytes = 128 * 128;     // one box: 128 rows x 128 bytes (a group pair)
constexpr int kMaxStages = 8;

// token operand bytes per group: 128 k x 8 token rows, or x 16 rows for 16 tokens
constexpr size_t token_group_bytes(int MT) { return MT > 8 ? 2048 : 1024; }
inline size_t tail_bytes(int MT, int G, int stages) {
    return (size_t)G * token_group_bytes(MT) + (((size_t)G * MT * 8 + 15) / 16) * 16 +
           (size_t)(2 * stages + 3 * kPSlots) * 8 + 16;
}
inline size_t smem_bytes(int MT, int K, int stages) {
    return (size_t)stages * kStageBytes + tail_bytes(MT, K / kGroup, stages);
}

// B byte order: MMA k-slot kappa of a group holds code k(kappa), where
//   u = kappa / 32, quad lane v = (kappa / 8) % 4, h = (kappa / 4) % 2, b = kappa % 4,
//   k(kappa) = 32 v + 8 u + 2 b + h
// (the A side: lane v of a quad holds codes 32 v .. 32 v + 31 of its rows;
// word u, nibble half h, byte b; the 16x256b store puts lo / hi of word u in
// columns 8 u + 2 v + {0, 1}).  So 4 consecutive k-slots are nibble half h of
// one activation word.
__device__ __forceinline__ uint32_t e4m3_of_signed_nibbles(uint32_t w, int h) {
    uint32_t r = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int q = (int32_t)((w >> (8 * b + 4 * h)) << 28) >> 28;
        const uint32_t e = q < 0 ? (0x80u | (uint32_t)(-q)) : (uint32_t)q;
        r |= e << (8 * b);
    }
    return r;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ xq,
                        const float *__restrict__ sx, const int32_t *__restrict__ qs,
                        const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y, int ldy,
                        int32_t *__restrict__ dbg_I, int32_t *__restrict__ st, int S, uint32_t wait_limit,
                        int stall) {
    static_assert(MT == 1 || MT == 2 || MT == 4 || MT == 8 || MT == 16, "token columns per CTA");
    constexpr uint32_t kTokBytes = (uint32_t)token_group_bytes(MT);
    extern __shared__ __align__(1024) unsigned char smem[];
    const int G = K / kGroup, P = (G + 1) / 2;
    uint8_t *stages = smem;
    uint8_t *bsm = smem + (size_t)S * kStageBytes;
    float2 *sxq = reinterpret_cast<float2 *>(bsm + (size_t)G * kTokBytes);
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sxq) + (((size_t)G * MT * 8 + 15) / 16) * 16);
    uint64_t *st_full = bars, *st_empty = bars + S;
    uint64_t *full = bars + 2 * S, *done = full + kPSlots, *freed = done + kPSlots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(freed + kPSlots);
    __shared__ int timeout_flag;
    __shared__ uint64_t never;                 // nothing arrives here (the stall test)
    __shared__ uint64_t drain_bar;             // the MMAs issued have completed
    volatile int *timeout = &timeout_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qr = lane >> 2, qc = lane & 3;
    const int tok0 = blockIdx.y * MT;
    const int n_tiles = (N + 127) / 128;
    const int my_tiles = (int)blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int n_pairs = my_tiles * P;          // one box, one TMEM pair slot each
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (*timeout) return false;
        if (umma::mbar_wait(bar, parity, wait_limit)) return true;
        *timeout = 1;
        return false;
    };

    if (threadIdx.x == 0) {
        *timeout = 0;
        for (int i = 0; i < S; ++i) {
            umma::mbar_init(&st_full[i], 1);
            umma::mbar_init(&st_empty[i], kConvWarps);
        }
        for (int s = 0; s < kPSlots; ++s) {
            umma::mbar_init(&full[s], kConvWarps);
            umma::mbar_init(&done[s], 1);
            umma::mbar_init(&freed[s], kEpiWarps);
        }
        umma::mbar_init(&never, 1);
        umma::mbar_init(&drain_bar, 1);
        umma::mbar_fence_init();
    }
    if (warp == kMmaWarp) umma::tmem_alloc(tmem_slot, kTmemCols);
    if (warp == kProducerWarp && lane == 0) umma::prefetch_tmap(&tmap);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    pdl_launch_dependents();

    // producer cursor over boxes (tile step, group pair)
    int pb = 0, pstep = 0, ppair = 0;
    auto issue_box = [&]() -> bool {
        const int slot = pb % S;
        if (pb >= S && !wait(&st_empty[slot], (uint32_t)(((pb / S) + 1) & 1))) return false;
        umma::mbar_arrive_expect_tx(&st_full[slot], kStageBytes);
        umma::tma_load_2d(stages + (size_t)slot * kStageBytes, &tmap, ppair * 128,
                          (blockIdx.x + pstep * gridDim.x) * 128, &st_full[slot]);
        ++pb;
        if (++ppair == P) {
            ppair = 0;
            ++pstep;
        }
        return true;
    };
    // the first boxes before the dependency wait: weights are immutable
    if (warp == kProducerWarp && lane == 0)
        while (pb < n_pairs && pb < S)
            if (!issue_box()) break;
    pdl_wait();

    // token operand: zero rows, then the real tokens' words
    for (int i = threadIdx.x; i < G * (int)(kTokBytes / 16); i += kThreads)
        reinterpret_cast<uint4 *>(bsm)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const int mt_real = min(MT, M - tok0);
    const uint32_t *xw = reinterpret_cast<const uint32_t *>(xq);
    for (int i = threadIdx.x; i < G * mt_real * 32; i += kThreads) {
        // (group g, token t, k-chunk kc, word j of the chunk)
        const int g = i / (mt_real * 32), rem = i - g * (mt_real * 32);
        const int t = rem >> 5, kc = (rem >> 2) & 7, j = rem & 3;
        const int c = 4 * kc + j;                         // 4-byte column of the group row
        const int u = c >> 3, v = (c & 7) >> 1, h = c & 1;
        const uint32_t w = xw[(size_t)(tok0 + t) * (K / 8) + g * 16 + 4 * v + u];
        // rows 0..7 of the chunk's core matrix, rows 8..15 in a second one 1024 bytes on
        reinterpret_cast<uint32_t *>(bsm + (size_t)g * kTokBytes + (t >> 3) * 1024 + kc * 128 + (t & 7) * 16)[j] =
            e4m3_of_signed_nibbles(w, h);
    }
    for (int i = threadIdx.x; i < G * MT; i += kThreads) {
        const int g = i / MT, t = i - g * MT, m = tok0 + t;
        sxq[i] = m < M ? make_float2(sx[(size_t)m * G + g], (float)qs[(size_t)m * G + g]) : make_float2(0.f, 0.f);
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tbase = *tmem_slot;
    int issued = 0;                            // pairs whose MMAs were issued (MMA lane 0)

    if (warp == kProducerWarp) {
        // ---- TMA producer ----
        if (lane == 0)
            while (pb < n_pairs)
                if (!issue_box()) break;
    } else if (warp == kMmaWarp) {
        // ---- MMA issuer: per pair, 4 MMAs per group present ----
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(0, 0, 128, 16);
            const uint32_t b0 = umma::smem_addr(bsm);
            if (stall) wait(&never, 0);
            int pp = 0;
            for (int p = 0; p < n_pairs; ++p) {
                const int s = p % kPSlots;
                if (!wait(&full[s], (uint32_t)((p / kPSlots) & 1))) break;
                umma::fence_after_sync();
                const int ng = 2 * pp + 1 < G ? 2 : 1;
                for (int gi = 0; gi < ng; ++gi) {
                    const uint32_t bg = b0 + (uint32_t)(2 * pp + gi) * kTokBytes;
                    // token rows 8..15: the second core-matrix row (16 tokens), else
                    // rows 0..7 again through a zero stride (ignored)
                    constexpr uint32_t kSbo = MT > 8 ? 1024 : 0;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma::mma_e4m3_ta(tbase + kDcol + 32 * s + 16 * gi, tbase + kAcol + 64 * s + 32 * gi + 8 * kk,
                                          umma::smem_desc(bg + kk * 256, 128, kSbo), idesc, kk > 0 ? 1u : 0u);
                }
                umma::mma_commit(&done[s]);
                ++issued;
                if (++pp == P) pp = 0;
            }
        }
    } else if (warp < kConvWarps) {
        // ---- converters: stage -> E4M3 bytes -> TMEM A slot (16 rows per warp) ----
        const int quad = warp & 3, half = warp >> 2;
        const uint32_t ta0 = tbase + kAcol + ((uint32_t)(32 * quad + 16 * half) << 16);
        const int r0 = 32 * quad + 16 * half + qr;                 // row % 8 = qr
        int pp = 0;
        for (int p = 0; p < n_pairs; ++p) {
            const int slot = p % S, s = p % kPSlots;
            if (!wait(&st_full[slot], (uint32_t)((p / S) & 1))) break;
            if (p >= kPSlots && !wait(&freed[s], (uint32_t)(((p / kPSlots) + 1) & 1))) break;
            umma::fence_after_sync();
            const uint8_t *stg = stages + (size_t)slot * kStageBytes;
            const int ng = 2 * pp + 1 < G ? 2 : 1;
            for (int gi = 0; gi < ng; ++gi) {
                const uint32_t pos = (uint32_t)(((4 * gi + qc) ^ qr) << 4);   // 128-byte swizzle
                const uint4 a = *reinterpret_cast<const uint4 *>(stg + (size_t)r0 * 128 + pos);
                const uint4 b = *reinterpret_cast<const uint4 *>(stg + (size_t)(r0 + 8) * 128 + pos);
                const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
                const uint32_t ta = ta0 + 64 * s + 32 * gi;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    umma::tmem_st16x256(ta + 8 * u, wa[u] & 0x0F0F0F0Fu, (wa[u] >> 4) & 0x0F0F0F0Fu,
                                        wb[u] & 0x0F0F0F0Fu, (wb[u] >> 4) & 0x0F0F0F0Fu);
            }
            umma::tmem_st_wait();
            umma::fence_before_sync();
            // the stage's next contents come by TMA (the async proxy): this
            // thread's reads of it are fenced against that before its release
            umma::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                umma::mbar_arrive(&full[s]);
                umma::mbar_arrive(&st_empty[slot]);
            }
            if (++pp == P) pp = 0;
        }
    } else {
        // ---- epilogue: thread = TMEM lane = output row of the tile ----
        const int q = warp - kConvWarps;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int erow = 32 * q + lane;
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
        // scale words of the next pair (rows past N read row 0)
        int zstep = 0, zpp = 0;
        // (both words in one 8-byte load when G is even and sz 8-byte aligned)
        const bool z64 = (G % 2) == 0 && (reinterpret_cast<uintptr_t>(sz) & 7) == 0;
        auto zload = [&](uint32_t &z0, uint32_t &z1) {
            const int n = (blockIdx.x + zstep * gridDim.x) * 128 + erow;
            const uint32_t *zp = sz + (size_t)(n < N ? n : 0) * G + 2 * zpp;
            if (z64) {
                const uint2 w = __ldg(reinterpret_cast<const uint2 *>(zp));
                z0 = w.x;
                z1 = w.y;
            } else {
                z0 = __ldg(zp);
                z1 = 2 * zpp + 1 < G ? __ldg(zp + 1) : 0u;
            }
            if (++zpp == P) {
                zpp = 0;
                ++zstep;
            }
        };
        uint32_t za = 0, zb = 0;
        if (n_pairs > 0) zload(za, zb);
        int pp = 0, step = 0;
        for (int p = 0; p < n_pairs; ++p) {
            const int s = p % kPSlots;
            const int ng = 2 * pp + 1 < G ? 2 : 1;
            if (!wait(&done[s], (uint32_t)((p / kPSlots) & 1))) break;
            umma::fence_after_sync();
            const uint32_t zw[2] = {za, zb};
            if (p + 1 < n_pairs) zload(za, zb);
            const int n = (blockIdx.x + step * gridDim.x) * 128 + erow;
            // the two groups' columns one after the other (registers for 16
            // tokens); the slot is freed once both are read
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                if (gi == 1 && ng == 1) break;
                uint32_t dg[MT];
                umma::tmem_ld_cols<MT>(tbase + kDcol + 32 * s + 16 * gi + lane_base, dg);
                umma::tmem_ld_wait();
                if (gi == ng - 1) {                        // once per pair, after its last read
                    umma::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) umma::mbar_arrive(&freed[s]);
                }
                const int g = 2 * pp + gi;
                const float zf = __half2float(__ushort_as_half((uint16_t)(zw[gi] >> 16)));
                const float sf = __half2float(__ushort_as_half((uint16_t)(zw[gi] & 0xFFFF)));
                // no branch inside the plain loop: the tokens' loads and FMAs
                // interleave (the debug output takes its own loop)
                if (dbg_I == nullptr) {
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float2 xv = sxq[g * MT + t];
                        const float I = __fmaf_rn(__uint_as_float(dg[t]), 262144.0f, -(zf * xv.y));
                        acc[t] = __fmaf_rn(I, __fmul_rn(xv.x, sf), acc[t]);
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float2 xv = sxq[g * MT + t];
                        const float I = __fmaf_rn(__uint_as_float(dg[t]), 262144.0f, -(zf * xv.y));
                        acc[t] = __fmaf_rn(I, __fmul_rn(xv.x, sf), acc[t]);
                        if (n < N && tok0 + t < M) dbg_I[((size_t)(tok0 + t) * N + n) * G + g] = (int32_t)I;
                    }
                }
            }
            if (++pp == P) {
                if (n < N) {
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        if (tok0 + t < M) y[(size_t)(tok0 + t) * ldy + n] = float_to_bf16_bits(acc[t]);
                }
#pragma unroll
                for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
                pp = 0;
                ++step;
            }
        }
    }

    // after a timeout: let this CTA's copies and MMAs in flight finish (bounded)
    // before the shared and tensor memory are released.  The producer stopped
    // issuing at the timeout, so at most S boxes are in flight, one per
    // stage; the MMA issuer's last commit covers all its MMAs.
    __syncthreads();
    if (*timeout) {
        if (warp == kProducerWarp && lane == 0)
            for (int b = max(0, pb - S); b < pb; ++b)
                umma::mbar_wait(&st_full[b % S], (uint32_t)((b / S) & 1), kWaitLimit);
        if (warp == kMmaWarp && lane == 0 && issued > 0) {
            umma::mma_commit(&drain_bar);
            umma::mbar_wait(&drain_bar, 0, kWaitLimit);
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *timeout) flag(st, QSPEC_ERR_TIMEOUT);
    if (warp == kMmaWarp) umma::tmem_free(tbase, kTmemCols);
}

template <int MT>
int launch(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed, const uint32_t *sz, int M,
           int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *dev_status, cudaStream_t stream,
           uint32_t wait_limit, int stall) {
    constexpr size_t kBudget = 220 * 1024;
    const int G = K / kGroup;
    const size_t tail = tail_bytes(MT, G, kMaxStages);
    if (tail + 2 * kStageBytes > kBudget) return QSPEC_ERR_SHAPE;
    const int S = (int)std::min<size_t>(kMaxStages, (kBudget - tail) / kStageBytes);
    CUtensorMap tmap;
    int rc = weight_tmap(&tmap, packed, N, K, 128);
    if (rc) return QSPEC_ERR_SHAPE;
    auto kern = w4a4_gemv_tc_kernel<MT>;
    rc = smem_limit_once(reinterpret_cast<const void *>(kern), (int)kBudget);
    if (rc) return rc;
    const int n_tiles = (N + 127) / 128, token_tiles = (M + MT - 1) / MT;
    const int per_col = std::max(1, sm_count() / token_tiles);
    dim3 grid((unsigned)std::min(n_tiles, per_col), (unsigned)token_tiles);
    return launch_pdl("qspec_linear_w4a4", kern, grid, dim3(kThreads), smem_bytes(MT, K, S), stream, tmap, xq, sx,
                      qs, sz, M, N, K, y, ldy, dbg_I, dev_status, S, wait_limit, stall);
}

}  // namespace tg

}  // namespace

// Decode-sized W4A4 on the tensor cores (M <= 16): QSPEC_OK, or
// QSPEC_ERR_SHAPE before any launch when the shape does not suit the kernel.
int launch_w4a4_gemv_tc(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                        const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I,
                        int32_t *dev_status, cudaStream_t stream, uint32_t wait_limit, int stall) {
    // 3..16 tokens (one and two tokens have their own kernels)
    if (M < 3 || M > 16) return QSPEC_ERR_SHAPE;
    if (M <= 4)
        return tg::launch<4>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, stream, wait_limit, stall);
    if (M <= 8)
        return tg::launch<8>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, stream, wait_limit, stall);
    return tg::launch<16>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, dev_status, stream, wait_limit, stall);
}

}  // namespace qspec
