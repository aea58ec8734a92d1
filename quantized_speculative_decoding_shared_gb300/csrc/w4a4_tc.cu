// w4a4_tc.cu -- a3, W4A4 linear on the Blackwell tensor cores for larger M
// (draft passes of large batches, prefill; also 13..32 tokens at large K,
// where the warp-MMA kernel would hold one token per CTA).
//
// QSPEC summary page, background terms: 4-bit activations times 4-bit
// weights, products accumulated exactly (INT32 in the pages' wording), then
// scaled to 16 bits.  Bit-exact definition (the same as the small-M kernels
// and the CPU oracle):
//   I[m][n][g] = sum_{k in g} q (W - z) ; acc = fmaf((float) I, sx * s, acc)
//   for g ascending from acc = 0 ; y = bf16_rn(acc).
//
// sm_103a has no integer tcgen05 MMA, so the products run as
// tcgen05.mma kind::f8f6f4 on E4M3 bytes that hold the integers exactly up
// to a power of two: a byte b in 0..15 read as E4M3 is b * 2^-9 (subnormal
// below 8, exponent 1 above), so a weight code needs no table -- its nibble
// is the byte -- and a token's q in [-8, 7] is the byte |q| with the sign
// bit set for q < 0.  Every product is c q 2^-18 with |c q| <= 120 and every
// partial sum of a group stays below 2^14 * 2^-18, so the fp32 accumulator
// holds D = 2^-18 sum q W exactly; the epilogue forms I = D 2^18 - z qs
// exactly in fp32 and folds it.  Inside each 8-wide k block both operands
// keep the even k first (w & 0x0F0F0F0F) and the odd k after
// ((w >> 4) & 0x0F0F0F0F): the MMA sums over k in any order common to both.
//
// Operands and roles (one CTA: 128 output channels x BN tokens of Y^T):
//   - the packed weight codes arrive by TMA, 128 channels x 128 bytes (two
//     groups) per box, 128-byte swizzle, into a ring of four boxes whose
//     first entries go out before the dependency wait (the weights are
//     immutable); warps 0-3 (thread = TMEM lane = channel) split each word
//     into its even- and odd-k bytes and store the group's 128 bytes into
//     one of four A buffers in tensor memory (32 columns);
//   - warps 12-15 build the tokens' E4M3 bytes for a group from the packed
//     activation codes into a B stage in shared memory (K-major, 128-byte
//     swizzle: 16-byte chunk j of token row t at position j ^ (t % 8));
//   - warps 16-17, lane 0 of each, issue the 4 MMAs (M = 128, N = BN,
//     K = 32) of every other group (a thread that issued MMAs waits for them
//     on its own next shared-memory access); each group has its own TMEM
//     accumulator, in batches of NB groups (4 at up to 32 tokens, 2 at up to
//     64, else 1) and two batches in flight;
//   - warps 4-11, two warpgroups on the same TMEM lanes with half of the
//     token columns each: per batch one barrier round, then per group TMEM ->
//     registers, I and the ordered fold in packed f32x2; finally bf16 (one
//     round per group cost ~1 us at 32 tokens, mostly barrier, wait and
//     scale-load latency);
//   - warp 18, lane 0, issues the code boxes.
// When the 128-channel tiles alone would leave SMs idle, a cluster of C CTAs
// (2 or 4) splits a tile's groups.  The fold must still run over all groups
// in ascending order, so no rank folds its own part: each stores its groups'
// exact I (|I| <= 128 * 8 * 15 fits 16 bits) in shared memory, and after a
// cluster barrier every rank folds a slice of the tile's outputs over all
// groups, reading the peers' I through distributed shared memory, then a
// second barrier keeps every rank's I alive until all have read.
// Bounded waits everywhere (the limit is a kernel argument; a test can also
// make an MMA issuer wait on a barrier nothing arrives at).  After a timeout
// (QSPEC_ERR_TIMEOUT) every role leaves its loop -- the epilogue warpgroups
// together, through a barrier that ORs their failure flags, since they also
// meet at a named barrier -- the code copies and MMAs in flight are drained
// with bounded waits, and the tensor memory is freed (even if a drain ran
// out: the next kernel on the SM would otherwise wait for it without bound).
#include <algorithm>
#include <type_traits>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

constexpr int kTileN = 128;                // output channels per CTA (MMA M)
constexpr int kAtom = 128;                 // bytes of K per row per group (E4M3)
constexpr int kConv = 128, kEpilogue = 256, kBld = 128;
constexpr int kEpiWarp0 = kConv / 32, kBldWarp0 = kEpiWarp0 + kEpilogue / 32;
constexpr int kMmaWarp = kBldWarp0 + kBld / 32, kTmaWarp = kMmaWarp + 2;   // two issuer warps
constexpr int kThreads = (kTmaWarp + 1) * 32;
constexpr int kCodeBox = kTileN * kAtom;   // packed codes of two groups for 128 channels
constexpr int kSC = 4;                     // code boxes in the ring
constexpr int kSA = 4;                     // A buffers in TMEM (32 columns: one group)

template <int BN>
constexpr int stage_bytes() { return BN * kAtom; }            // the tokens' bytes of one group
template <int BN>
constexpr int n_stages() {                 // even: each issuer then uses its own stages
    return std::min(4, (200 * 1024 - kSC * kCodeBox) / stage_bytes<BN>()) & ~1;
}

// K-major 128-byte-swizzle descriptor: start address, leading offset unused
// (16 bytes), 1024 bytes between 8-row groups, version 1, swizzle mode 2
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// four two's-complement q (one per byte, low nibble) -> E4M3 bytes of q 2^-9
__device__ __forceinline__ uint32_t e4m3_q4(uint32_t b) {
    const uint32_t s = (b >> 3) & 0x01010101u;                 // 1 where q < 0
    const uint32_t mag = (b ^ (s * 0x0Fu)) + s;                // |q| in 0..8, no carry out of a byte
    return mag | (s << 7);
}

__device__ __forceinline__ uint64_t f2(float a, float b) {
    return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// accumulator columns of one group and groups per epilogue batch: the
// epilogue takes NB groups per barrier round, and two batches of NB
// accumulators (256 TMEM columns) let the MMAs run a batch ahead of it
template <int BN>
constexpr int acc_cols() { return BN <= 32 ? 32 : BN <= 64 ? 64 : 128; }
template <int BN>
constexpr int batch_groups() { return 128 / acc_cols<BN>(); }

template <int BN>
struct Ctl {
    float esx[2][batch_groups<BN>() * BN];   // epilogue-owned: sx of the batch's tokens, [group][token]
    float enqs[2][batch_groups<BN>() * BN];  // -qs as float (exact)
    uint64_t afull[kSA], aempty[kSA];  // A buffers: stored / read by the MMAs
    uint64_t bfull[4], bempty[4];      // token stages: built / read
    uint64_t cfull[kSC], cempty[kSC];  // code boxes: landed / read by every converter
    uint64_t accf[2], acce[2];         // accumulator batches: computed / drained
    uint64_t drain[2];                 // after a timeout: each issuer's MMAs in flight have finished
    uint64_t never;                    // nothing arrives here (the stall test)
    uint32_t tmem;
    int timeout;
};

template <int BN>
constexpr size_t smem_total() {
    return (size_t)n_stages<BN>() * stage_bytes<BN>() + (size_t)kSC * kCodeBox + sizeof(Ctl<BN>) + 1024;
}

// kPlain: no debug output -- the folds then have no branch inside and fewer
// live registers (no spills at up to 48 tokens)
template <int BN, bool kPlain>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_umma_kernel(const __grid_constant__ CUtensorMap tw, const uint8_t *__restrict__ xq,
                     const float *__restrict__ sx, const int32_t *__restrict__ qs, const uint32_t *__restrict__ sz,
                     int M, int N, int K, uint16_t *__restrict__ y, int ldy, int32_t *__restrict__ dbg_I,
                     int32_t *st, int C, uint32_t wait_limit, int stall) {
    constexpr int S = n_stages<BN>();
    constexpr int kStage = stage_bytes<BN>();
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128 && S >= 2, "token tile");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // stages 1024-aligned (the swizzle pattern is a function of the address)
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *codes = stages + (size_t)S * kStage;                 // kSC boxes of kCodeBox bytes
    Ctl<BN> &sm = *reinterpret_cast<Ctl<BN> *>(codes + (size_t)kSC * kCodeBox);
    // split groups: this rank's exact I, int16 [group][channel][token]
    int16_t *ibuf = reinterpret_cast<int16_t *>(reinterpret_cast<uint8_t *>(&sm) + ((sizeof(Ctl<BN>) + 15) & ~size_t(15)));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = C > 1 ? (int)umma::cluster_rank() : 0;
    const int n0 = (blockIdx.x / C) * kTileN, t0 = blockIdx.y * BN;
    const int G = K / kGroup;
    const int g_lo = (int)(((long long)rank * G) / C), g_hi = (int)(((long long)(rank + 1) * G) / C);
    const int NG = g_hi - g_lo;                          // this CTA's groups
    // TMEM: two batches of NB accumulators of kBuf columns (256 columns),
    // then kSA A buffers of 32
    constexpr uint32_t kBuf = acc_cols<BN>();
    constexpr int NB = batch_groups<BN>();
    constexpr uint32_t kAcol = 2 * NB * kBuf;
    constexpr uint32_t kCols = 512;
    static_assert(kAcol + 32 * kSA <= kCols && NB * BN <= kEpilogue, "tensor memory plan");
    const int NBt = (NG + NB - 1) / NB;                  // batches

    if (warp == 0) umma::tmem_alloc(&sm.tmem, kCols);
    if (tid == 0) {
        for (int s = 0; s < kSA; ++s) {
            umma::mbar_init(&sm.afull[s], kConv);
            umma::mbar_init(&sm.aempty[s], 1);
        }
        for (int s = 0; s < S; ++s) {
            umma::mbar_init(&sm.bfull[s], kBld);
            umma::mbar_init(&sm.bempty[s], 1);
        }
        for (int c = 0; c < kSC; ++c) {
            umma::mbar_init(&sm.cfull[c], 1);
            umma::mbar_init(&sm.cempty[c], kConv);
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(&sm.accf[b], NB >= 2 ? 2 : 1);     // a commit from each issuer with a part in the batch
            umma::mbar_init(&sm.acce[b], kEpilogue);
            umma::mbar_init(&sm.drain[b], 1);
        }
        umma::mbar_init(&sm.never, 1);
        sm.timeout = 0;
        umma::mbar_fence_init();
    }
    if (warp == kTmaWarp && lane == 0) umma::prefetch_tmap(&tw);
    pdl_launch_dependents();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    bool issued = false;                          // MMAs issued (issuer lane 0)
    int copies = 0;                               // code boxes issued (copy lane 0)
    auto timed_out = [&]() { return *reinterpret_cast<volatile int *>(&sm.timeout) != 0; };
    auto give_up = [&]() { atomicExch(&sm.timeout, 1); };

    if (warp < kEpiWarp0) {
        // ------------------------------------------------------ weight converters
        // thread = channel r = TMEM lane; its 64 code bytes of a group come
        // from the code box (row r, 16-byte chunks 4 (l % 2) .. + 3, 128-byte
        // swizzle); rows past N arrive as zeros
        const int r = tid;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        // group l's 128 codes -> 32 words of bytes (per code word, even k then
        // odd k); false if its code box did not arrive in time
        auto convert = [&](int l, uint32_t (&v)[32]) {
            const int c = (l >> 1) % kSC;
            if ((l & 1) == 0 && (timed_out() || !umma::mbar_wait(&sm.cfull[c], ((l >> 1) / kSC) & 1, wait_limit)))
                return false;
            const uint8_t *crow = codes + (size_t)c * kCodeBox + (size_t)r * kAtom;
            uint4 cw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                cw[u] = *reinterpret_cast<const uint4 *>(crow + (((4 * (l & 1) + u) ^ (r & 7)) << 4));
            // the box's next contents come by TMA (the async proxy): these
            // reads are fenced against it before the box is released
            if ((l & 1) == 1 || l + 1 == NG) {
                umma::fence_proxy_async();
                umma::mbar_arrive(&sm.cempty[c]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w4[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[8 * u + 2 * q] = w4[q] & 0x0F0F0F0Fu;
                    v[8 * u + 2 * q + 1] = (w4[q] >> 4) & 0x0F0F0F0Fu;
                }
            }
            return true;
        };
        // group l from cur into its A buffer; the next group is loaded and
        // unpacked into nxt while the copy to tensor memory is in flight
        auto step = [&](int l, const uint32_t (&cur)[32], uint32_t (&nxt)[32]) {
            const int sa = l % kSA;
            if (l >= kSA && (timed_out() || !umma::mbar_wait(&sm.aempty[sa], ((l / kSA) - 1) & 1, wait_limit)))
                return false;
            umma::fence_after_sync();
            umma::tmem_st32(tmem + lane_off + kAcol + (uint32_t)(sa * 32), cur);
            const bool next_ok = l + 1 >= NG || convert(l + 1, nxt);
            umma::tmem_st_wait();
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.afull[sa]);
            return next_ok;
        };
        uint32_t va[32], vb[32];
        bool ok = NG == 0 || convert(0, va);
        for (int l = 0; ok && l < NG; l += 2) {
            ok = step(l, va, vb);
            if (ok && l + 1 < NG) ok = step(l + 1, vb, va);
        }
        if (!ok) give_up();
    } else if (warp < kBldWarp0) {
        // ------------------------------------------------------------ epilogue
        pdl_wait();
        constexpr int kHalf = BN / 2;                 // token columns per warpgroup
        constexpr int kW = kHalf % 16 == 0 ? 16 : 8;
        const int eq = warp & 3;                      // TMEM lanes 32 eq .. 32 eq + 31
        const int eh = (warp - kEpiWarp0) >> 2;       // column half
        const int et = tid - kConv;                   // 0 .. 255
        const int n = n0 + eq * 32 + lane;
        const bool row_ok = n < N;
        const uint64_t k18 = f2(262144.0f, 262144.0f);
        uint64_t acc[kHalf / 2];
#pragma unroll
        for (int i = 0; i < kHalf / 2; ++i) acc[i] = 0;
        bool ok = true;
        // thread et < NB * BN loads the sx, qs of token t0 + et % BN, group
        // et / BN of the next batch, one batch ahead
        const int tt = et % BN, tj = et / BN;
        const bool tok_ok = et < NB * BN && t0 + tt < M;
        const float *sxp = sx + (size_t)(tok_ok ? t0 + tt : 0) * G + g_lo + tj;
        const int32_t *qsp = qs + (size_t)(tok_ok ? t0 + tt : 0) * G + g_lo + tj;
        float sx_n = tok_ok && tj < NG ? sxp[0] : 0.0f;
        int32_t qs_n = tok_ok && tj < NG ? qsp[0] : 0;
        // the channel's scale words, one batch ahead
        const uint32_t *szp = sz + (size_t)(row_ok ? n : 0) * G + g_lo;
        uint32_t szn[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) szn[j] = 0u;
        // the batch's NB scale words of the row in one vector load when aligned
        // (one request instead of NB: 32-token LM head 152 -> 131 us)
        const bool szvec = NB >= 2 && (G % NB) == 0 && (g_lo % NB) == 0 &&
                           (reinterpret_cast<uintptr_t>(sz) & (4 * NB - 1)) == 0;
        auto load_sz = [&](int l0) {
            if (!row_ok) return;
            if (szvec && l0 + NB <= NG) {
                if constexpr (NB == 4) {
                    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(szp + l0));
                    szn[0] = w.x;
                    szn[1] = w.y;
                    szn[2] = w.z;
                    szn[3] = w.w;
                } else if constexpr (NB == 2) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(szp + l0));
                    szn[0] = w.x;
                    szn[1] = w.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < NB; ++j) szn[j] = l0 + j < NG ? __ldg(szp + l0 + j) : 0u;
            }
        };
        load_sz(0);
        for (int b = 0; b < NBt; ++b) {
            const int set = b & 1, lb = b * NB, nb = min(NB, NG - lb);
            // the batch's token scales into the epilogue's own double buffer;
            // the barrier also orders this write after every epilogue
            // thread's reads of the same buffer two batches ago, and tells
            // every epilogue thread whether any of them has given up (all
            // leave together)
            if (et < NB * BN) {
                sm.esx[set][et] = sx_n;
                sm.enqs[set][et] = -(float)qs_n;
                if (tok_ok && lb + NB + tj < NG) {
                    sx_n = sxp[lb + NB];
                    qs_n = qsp[lb + NB];
                }
            }
            uint32_t any_failed;
            asm volatile(
                "{.reg .pred p, q; setp.eq.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q;}\n"
                : "=r"(any_failed)
                : "r"(ok ? 1u : 0u), "r"(kEpilogue)
                : "memory");
            if (any_failed) break;
            if (timed_out() || !umma::mbar_wait(&sm.accf[set], (b >> 1) & 1, wait_limit)) {
                give_up();
                ok = false;
                continue;                             // to the barrier, where all leave
            }
            umma::fence_after_sync();
            uint32_t szc[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                szc[j] = szn[j];
            }
            load_sz(lb + NB);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                if (j >= nb) break;
                const int l = lb + j, g = g_lo + l;
                const float sn = __half2float(__ushort_as_half((uint16_t)(szc[j] & 0xFFFF)));
                const float zn = __half2float(__ushort_as_half((uint16_t)(szc[j] >> 16)));
                const uint64_t s2 = f2(sn, sn), z2 = f2(zn, zn);
                const float *esx = &sm.esx[set][j * BN];
                const float *enqs = &sm.enqs[set][j * BN];
                // the plain fold has no branch inside, so the pairs' loads and
                // packed operations interleave (a branch per pair measured
                // 1.4x slower at 32 and 64 tokens); the split (cross-rank I)
                // and debug paths take the general loop
                // mode 0: one rank, the ordered fold; mode 1: split groups,
                // the exact I kept for the cross-rank fold; mode 2: either,
                // with the debug output
                auto fold = [&](auto mode_tag) {
                    constexpr int kMode = decltype(mode_tag)::value;
#pragma unroll
                    for (int c0 = 0; c0 < kHalf; c0 += kW) {
                        uint32_t v[kW];
                        const uint32_t ta = tmem + ((uint32_t)(eq * 32) << 16) +
                                            (uint32_t)((set * NB + j) * kBuf + eh * kHalf + c0);
                        umma::tmem_ld_cols<kW>(ta, *reinterpret_cast<uint32_t(*)[kW]>(v));
                        umma::tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < kW; jj += 2) {
                            const int t = eh * kHalf + c0 + jj;
                            // I = D 2^18 - z qs (exact), c = sx * s, acc = fma(I, c, acc)
                            const uint64_t nqs2 = *reinterpret_cast<const uint64_t *>(&enqs[t]);
                            const uint64_t I2 =
                                fma2(f2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])), k18, mul2(z2, nqs2));
                            if constexpr (kMode == 0) {
                                const uint64_t sx2 = *reinterpret_cast<const uint64_t *>(&esx[t]);
                                acc[(c0 + jj) / 2] = fma2(I2, mul2(sx2, s2), acc[(c0 + jj) / 2]);
                            } else if constexpr (kMode == 1) {
                                const int row = eq * 32 + lane;
                                ibuf[((size_t)l * kTileN + row) * BN + t] = (int16_t)__uint_as_float((uint32_t)I2);
                                ibuf[((size_t)l * kTileN + row) * BN + t + 1] =
                                    (int16_t)__uint_as_float((uint32_t)(I2 >> 32));
                            } else {
                                if (C == 1) {
                                    const uint64_t sx2 = *reinterpret_cast<const uint64_t *>(&esx[t]);
                                    acc[(c0 + jj) / 2] = fma2(I2, mul2(sx2, s2), acc[(c0 + jj) / 2]);
                                } else {              // kept for the cross-rank fold
                                    const int row = eq * 32 + lane;
                                    ibuf[((size_t)l * kTileN + row) * BN + t] = (int16_t)__uint_as_float((uint32_t)I2);
                                    ibuf[((size_t)l * kTileN + row) * BN + t + 1] =
                                        (int16_t)__uint_as_float((uint32_t)(I2 >> 32));
                                }
                                if (dbg_I != nullptr && row_ok) {
                                    const int m0 = t0 + t;
                                    if (m0 < M) dbg_I[((size_t)m0 * N + n) * G + g] = (int32_t)__uint_as_float((uint32_t)I2);
                                    if (m0 + 1 < M)
                                        dbg_I[((size_t)(m0 + 1) * N + n) * G + g] =
                                            (int32_t)__uint_as_float((uint32_t)(I2 >> 32));
                                }
                            }
                        }
                    }
                };
                if constexpr (!kPlain)
                    fold(std::integral_constant<int, 2>());
                else if (C == 1)
                    fold(std::integral_constant<int, 0>());
                else
                    fold(std::integral_constant<int, 1>());
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.acce[set]);
        }
        if (C == 1 && ok && row_ok) {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
                const int m = t0 + eh * kHalf + 2 * i;
                if (m < M) y[(size_t)m * ldy + n] = float_to_bf16_bits(__uint_as_float((uint32_t)acc[i]));
                if (m + 1 < M) y[(size_t)(m + 1) * ldy + n] = float_to_bf16_bits(__uint_as_float((uint32_t)(acc[i] >> 32)));
            }
        }
    } else if (warp < kMmaWarp) {
        // ------------------------------------------------------------ token builders
        // task = (token row t, 16-byte quarter u of the group's 64 code bytes):
        // 32 codes -> 32 E4M3 bytes, the 16-byte chunks 2 u and 2 u + 1 of row t
        pdl_wait();
        const int bt = tid - kBldWarp0 * 32;
        constexpr int kTasks = BN * 4, kPer = (kTasks + kBld - 1) / kBld;
        auto load = [&](int l, uint4 (&xv)[kPer]) {
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int task = bt + i * kBld, t = task >> 2, u = task & 3, m = t0 + t;
                xv[i] = (task < kTasks && m < M && l < NG)
                            ? __ldg(reinterpret_cast<const uint4 *>(xq + (size_t)m * (K / 2) + (size_t)(g_lo + l) * 64) + u)
                            : make_uint4(0, 0, 0, 0);
            }
        };
        uint4 xn[kPer];
        load(0, xn);
        for (int l = 0; l < NG; ++l) {
            const int s = l % S;
            uint4 xv[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) xv[i] = xn[i];
            load(l + 1, xn);
            if (l >= S && (timed_out() || !umma::mbar_wait(&sm.bempty[s], ((l / S) - 1) & 1, wait_limit))) {
                give_up();
                break;
            }
            uint8_t *b = stages + (size_t)s * kStage;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int task = bt + i * kBld, t = task >> 2, u = task & 3;
                if (task >= kTasks) break;
                const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
                uint32_t e[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    e[2 * q] = e4m3_q4(w4[q] & 0x0F0F0F0Fu);
                    e[2 * q + 1] = e4m3_q4((w4[q] >> 4) & 0x0F0F0F0Fu);
                }
                uint8_t *row = b + (size_t)(t >> 3) * 1024 + (size_t)(t & 7) * 128;
                *reinterpret_cast<uint4 *>(row + (((2 * u) ^ (t & 7)) << 4)) = make_uint4(e[0], e[1], e[2], e[3]);
                *reinterpret_cast<uint4 *>(row + (((2 * u + 1) ^ (t & 7)) << 4)) = make_uint4(e[4], e[5], e[6], e[7]);
            }
            umma::fence_proxy_async();
            umma::mbar_arrive(&sm.bfull[s]);
        }
    } else if (warp < kTmaWarp) {
        // ------------------------------------------------------------ MMA issuers
        // issuer i takes groups l = i, i + 2, ...: A buffers and token stages
        // of parity i (kSA and S are even), so each barrier it polls is at
        // most one phase ahead of the last it saw; the accumulators of a batch
        // are reused only after the epilogue has drained the batch two back
        const int iss = warp - kMmaWarp;
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(0, 0, kTileN, BN);   // e4m3 x e4m3 -> f32
            if (stall && iss == 0 && !umma::mbar_wait(&sm.never, 0, wait_limit)) give_up();
            for (int b = 0; b < NBt; ++b) {
                // batch b: groups lb .. lb + nb - 1 into accumulator set b & 1;
                // with NB >= 2 both issuers take part (and commit) in every
                // batch, with NB = 1 the batch's one group belongs to issuer b & 1
                const int set = b & 1, lb = b * NB, nb = min(NB, NG - lb);
                if (NB == 1 && set != iss) continue;
                if (b >= 2 && (timed_out() || !umma::mbar_wait(&sm.acce[set], ((b >> 1) - 1) & 1, wait_limit))) {
                    give_up();
                    break;
                }
                bool failed = false;
                for (int l = lb + ((lb & 1) != iss ? 1 : 0); l < lb + nb; l += 2) {
                    const int sa = l % kSA, sb = l % S;
                    if (timed_out() || !umma::mbar_wait(&sm.afull[sa], (l / kSA) & 1, wait_limit) ||
                        !umma::mbar_wait(&sm.bfull[sb], (l / S) & 1, wait_limit)) {
                        failed = true;
                        break;
                    }
                    umma::fence_after_sync();
                    const uint64_t db = desc_sw128(umma::smem_addr(stages + (size_t)sb * kStage));
                    const uint32_t a0 = tmem + kAcol + (uint32_t)(sa * 32);
                    const uint32_t d = tmem + (uint32_t)((set * NB + (l - lb)) * kBuf);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // K = 32 bytes: 8 TMEM columns of A, +2 in B's address field
                        umma::mma_e4m3_ta(d, a0 + 8 * kk, db + 2 * kk, idesc, kk != 0 ? 1u : 0u);
                    umma::mma_commit(&sm.aempty[sa]);
                    umma::mma_commit(&sm.bempty[sb]);
                    issued = true;
                }
                if (failed) {
                    give_up();
                    break;
                }
                umma::mma_commit(&sm.accf[set]);   // arrives once this issuer's MMAs so far are done
                issued = true;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ code boxes
        if (lane == 0) {
            const int NP = (NG + 1) / 2;
            for (int p = 0; p < NP; ++p) {
                const int c = p % kSC;
                if (p >= kSC && (timed_out() || !umma::mbar_wait(&sm.cempty[c], ((p / kSC) - 1) & 1, wait_limit))) {
                    give_up();
                    break;
                }
                umma::mbar_arrive_expect_tx(&sm.cfull[c], (uint32_t)kCodeBox);
                umma::tma_load_2d(codes + (size_t)c * kCodeBox, &tw, (g_lo + 2 * p) * (kGroup / 2), n0, &sm.cfull[c]);
                copies = p + 1;
            }
        }
        __syncwarp();
    }
    umma::fence_before_sync();
    __syncthreads();
    // after a timeout, the copies and MMAs already issued finish (bounded
    // waits) before the shared and tensor memory are released; sm.timeout is
    // settled at this barrier
    if (sm.timeout) {
        if (warp == kTmaWarp && lane == 0)
            for (int p = std::max(0, copies - kSC); p < copies; ++p)
                umma::mbar_wait(&sm.cfull[p % kSC], (p / kSC) & 1, kWaitLimit);
        if (warp >= kMmaWarp && warp < kTmaWarp && lane == 0 && issued) {
            umma::mma_commit(&sm.drain[warp - kMmaWarp]);
            umma::mbar_wait(&sm.drain[warp - kMmaWarp], 0, kWaitLimit);
        }
        __syncthreads();
    }
    if (C > 1) {
        // every rank's I is complete; this rank folds channels
        // [rank * 128 / C, (rank + 1) * 128 / C) over all groups in ascending
        // order, each group's I read from the rank that computed it.  The
        // tokens' sx and the channels' s go to shared memory first (the code
        // ring is free now).
        umma::cluster_sync();
        const bool all_ok = !sm.timeout;
        const int rows = kTileN / C, r0 = rank * rows;
        float *sxs = reinterpret_cast<float *>(codes);            // [G][BN]
        float *ss = sxs + (size_t)BN * G;                          // [rows][G]
        if (warp >= kEpiWarp0 && warp < kBldWarp0 && all_ok) {
            const int et = tid - kConv;
            for (int i = et; i < BN * G; i += kEpilogue) {
                const int g = i / BN, t = i - g * BN, m = t0 + t;
                sxs[i] = m < M ? sx[(size_t)m * G + g] : 0.0f;
            }
            for (int i = et; i < rows * G; i += kEpilogue) {
                const int rr = i / G, g = i - rr * G, n = n0 + r0 + rr;
                ss[i] = n < N ? __half2float(__ushort_as_half((uint16_t)(__ldg(sz + (size_t)n * G + g) & 0xFFFF)))
                              : 0.0f;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kEpilogue) : "memory");
            // task = (channel, 8 consecutive tokens): one 16-byte read of the
            // eight I per group, four groups' reads in flight
            constexpr int kCh = BN / 8;
            for (int e = et; e < rows * kCh; e += kEpilogue) {
                const int rr = e / kCh, tb = (e - rr * kCh) * 8, row = r0 + rr, n = n0 + row;
                if (n >= N) continue;
                const float *sr = ss + (size_t)rr * G;
                float acc[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
                for (int q = 0; q < C; ++q) {
                    const int qlo = (int)(((long long)q * G) / C), qhi = (int)(((long long)(q + 1) * G) / C);
                    const int16_t *ib = &ibuf[(size_t)row * BN + tb];
                    for (int g = qlo; g < qhi; g += 4) {
                        uint4 I8[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            I8[u] = g + u < qhi ? umma::ld_peer_v4(ib + (size_t)(g + u - qlo) * kTileN * BN, (uint32_t)q)
                                                : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (g + u >= qhi) break;
                            const float s = sr[g + u];
                            const float *sxg = sxs + (size_t)(g + u) * BN + tb;
                            const uint32_t w[4] = {I8[u].x, I8[u].y, I8[u].z, I8[u].w};
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float I = (float)(int16_t)(uint16_t)(w[j >> 1] >> (16 * (j & 1)));
                                acc[j] = __fmaf_rn(I, __fmul_rn(sxg[j], s), acc[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (t0 + tb + j < M) y[(size_t)(t0 + tb + j) * ldy + n] = float_to_bf16_bits(acc[j]);
            }
        }
        umma::cluster_sync();                    // peers' I stay until every rank has read
    }
    if (tid == 0 && sm.timeout) flag(st, QSPEC_ERR_TIMEOUT);
    if (warp == 0) umma::tmem_free(tmem, kCols);
}

template <int BN>
int launch_bn(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed, const uint32_t *sz,
              int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st, cudaStream_t stream,
              uint32_t wait_limit, int stall) {
    CUtensorMap tw;
    // the packed codes: rows of K / 2 bytes, boxes of 128 bytes x 128 channels
    if (byte_tmap_sw128(&tw, packed, N, K / 2, (size_t)K / 2, kTileN)) return QSPEC_ERR_UNSUPPORTED;
    const int n_tiles = (N + kTileN - 1) / kTileN, token_tiles = (M + BN - 1) / BN, G = K / kGroup;
    // split the groups over a cluster of 4 (else 2) CTAs, one per SM, when
    // the tiles alone leave SMs idle and a rank's I fits in shared memory --
    // at 16-token tiles only: measured 74 -> 39 us (4096 x 14336) and 23 -> 17
    // us (4096 x 4096) at 16 tokens with 4 CTAs, 6144 x 4096 with 2 faster
    // than unsplit since the folds lost their per-element branches, but
    // slower at 32-token tiles (6144 x 4096: 23 -> 61 us)
    const size_t kIbufMax = 227 * 1024 - smem_total<BN>() - 16;
    int C = 1;
    if (BN == 16)
        for (int c : {4, 2})
        if (n_tiles * token_tiles * c <= sm_count() && 2 * c <= G &&
            (size_t)((G + c - 1) / c) * kTileN * BN * 2 <= kIbufMax &&
            (size_t)(BN + kTileN / c) * G * 4 <= (size_t)kSC * kCodeBox) {   // the fold's scale tables
            C = c;
            break;
        }
    const size_t ibuf = C > 1 ? (size_t)((G + C - 1) / C) * kTileN * BN * 2 + 16 : 0;
    const size_t smem = smem_total<BN>() + ibuf;
    if (smem > 227 * 1024) return QSPEC_ERR_SHAPE;
    dim3 grid((unsigned)(n_tiles * C), (unsigned)token_tiles);
    auto go = [&](auto kern) {
        int rc = smem_limit_once(reinterpret_cast<const void *>(kern), 227 * 1024);
        if (rc) return rc;
        if (C == 1)
            return launch_pdl("qspec_linear_w4a4", kern, grid, dim3(kThreads), smem, stream, tw, xq, sx, qs, sz, M, N,
                              K, y, ldy, dbg_I, st, C, wait_limit, stall);
        return launch_pdl_cluster("qspec_linear_w4a4", kern, grid, dim3(kThreads), smem, stream, C, tw, xq, sx, qs,
                                  sz, M, N, K, y, ldy, dbg_I, st, C, wait_limit, stall);
    };
    return dbg_I == nullptr ? go(&w4a4_umma_kernel<BN, true>) : go(&w4a4_umma_kernel<BN, false>);
}

}  // namespace

// Larger-M W4A4 on the tensor cores: below 256 tokens ceil(M / 128) token
// tiles of BN tokens (a multiple of 16, 16 ... 128); from 256 tokens the
// prefill kernel of w4a4_tc_wide.cu.
int launch_w4a4_tc(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                   const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st,
                   cudaStream_t stream, uint32_t wait_limit, int stall) {
    if (M >= 256)          // prefill-sized: the fold bounds it, see w4a4_tc_wide.cu
        return launch_w4a4_tc_wide(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
    // up to 32 tokens on layers with fewer 128-channel tiles than SMs: 16-token
    // tiles (twice the CTAs, the second token tile reading the weights out of
    // L2; 32 tokens: 4096 x 4096 22.5 -> 18.9 us, 4096 x 14336 63.9 -> 58.9 us,
    // but the larger layers slower)
    const int tiles = (M + 127) / 128, per = (M + tiles - 1) / tiles;
    const int bn = M <= 32 && (N + 127) / 128 < sm_count() ? 16 : (per + 15) / 16 * 16;
    switch (bn) {
        case 16: return launch_bn<16>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 32: return launch_bn<32>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 48: return launch_bn<48>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 64: return launch_bn<64>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 80: return launch_bn<80>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 96: return launch_bn<96>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        case 112: return launch_bn<112>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
        default: return launch_bn<128>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
    }
}

}  // namespace qspec
