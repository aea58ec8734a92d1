// w4a16_tc.cu -- a4, W4A16 linear on the Blackwell tensor cores for M > 16
// (verify passes of larger batches: M = B (gamma + 1) = 80 ... 288, prefill).
//
// QSPEC summary page, background terms: the 4-bit weights are dequantised
// for the matmul, W^ = s (W_INT4 - z), Y = X W^, with 16-bit activations;
// "QSPEC structure": the verify pass.
//
// The dequantisation is split so that nothing is rounded before the fp32
// accumulation: the tensor core multiplies the activations by the exact
// integers c - z (bf16 holds every integer in [-15, 15]) and sums one
// 128-wide group into a TMEM accumulator in fp32; the epilogue applies the
// group's scale, y += s * D_g, in fp32 registers.
//
// Operands:
//   - the activations (B) arrive by TMA in shared memory, two boxes of BN
//     tokens x 64 k per group, in the K-major layout with 128-byte swizzle
//     (rows of 64 bf16; 8-row groups 1024 bytes apart; the 16-byte chunk j of
//     row r at position j ^ (r % 8)), which the MMA reads directly;
//   - the packed codes arrive by TMA too, 128 channels x 128 bytes (two
//     groups) per box, into a ring of four boxes whose first entries go out
//     before the dependency wait (the weights are immutable); 8 warps convert
//     them, two threads per output channel, each 64 k of a group: the codes
//     of a word are split one per byte (even k, odd k), interleaved back into
//     k order and spread into the low bytes of bf16 lanes of 128.0 by byte
//     permutes, which gives the bf16 pairs (128 + c_2j, 128 + c_2j+1)
//     exactly; one exact bf16 subtraction of 128 + z leaves (c - z);
//   - the converted weights (A) go to tensor memory, not shared memory (lane
//     = output channel, column = a pair of consecutive k), and the MMA reads
//     them there: written and read in shared memory they would share its
//     bandwidth with the activations and the codes, and bound the kernel.
// One CTA computes a 128 (output channels) x BN (tokens) tile of Y^T:
//   warps 0-7   weight converters (warp w: TMEM lanes 32 (w % 4) .., k half w / 4)
//   warps 8-15  epilogue, two warpgroups on the same TMEM lanes, each with
//               half of the token columns: per group, TMEM -> registers,
//               y = fma(D, s, y) in packed f32x2; finally bf16
//   warps 16-17 lane 0 of each issues the 8 MMAs (K = 16) of every other
//               group, into its own TMEM accumulator, A from one of four TMEM
//               operand buffers (a thread that issued MMAs waits for them on
//               its own next shared-memory access, so one issuer alone would
//               leave the tensor core idle between groups)
//   warp 18     lane 0 issues the code boxes, lane 1 the activation boxes
// When the 128-channel tiles alone would leave SMs idle, a cluster of up to 8
// CTAs splits a tile's groups; each CTA keeps its fp32 partial sums, and
// rank 0 reads its peers' partials from distributed shared memory, adds them
// in rank order and stores bf16.
// Bounded waits everywhere (the limit is a kernel argument; a test can also
// make the MMA issuer wait on a barrier nothing arrives at).  After a
// timeout (QSPEC_ERR_TIMEOUT) every role leaves its loop, the activation
// copies and the MMAs issued are drained with bounded waits, and the tensor
// memory is freed -- even if a drain ran out (the next kernel on the SM would
// otherwise wait for it without bound); in that case the split-K reduction,
// which reuses the operand stages, is skipped.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

constexpr int kTileN = 128;              // output channels per CTA (MMA M)
constexpr int kAtom = 128;               // bytes of K per swizzle atom row (64 bf16)
constexpr int kConv = 256;               // converter threads: two per channel
constexpr int kEpilogue = 256;
constexpr int kMmaWarp = (kConv + kEpilogue) / 32, kTmaWarp = kMmaWarp + 2;   // two issuer warps
constexpr int kThreads = kConv + kEpilogue + 96;
constexpr int kCodeBox = kTileN * kAtom; // packed codes of two groups for 128 channels
constexpr int kSC = 4;                   // code boxes counted when sizing the token stages
constexpr int kSA = 4;                   // A operand buffers in TMEM (64 columns: one group)

template <int BN>
constexpr int stage_bytes() { return BN * 2 * kAtom; }       // activations of one group
template <int BN>
constexpr int n_stages() {   // even: each issuer then uses its own stages
    return std::min(4, (212 * 1024 - kSC * kCodeBox) / stage_bytes<BN>()) & ~1;
}

// Code boxes in the ring: whatever shared memory the token stages leave (up
// to 12 boxes, 24 groups in flight); with four boxes the DRAM latency of the
// copies set the pace.
template <int BN>
constexpr int ring_boxes() {
    return std::min(12, (227 * 1024 - 4096 - n_stages<BN>() * stage_bytes<BN>()) / kCodeBox);
}

__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// eight codes of a word (k = 0..7) -> 16 bytes of bf16 (c - z), natural k order:
// the codes one per byte (even k / odd k), interleaved in k order, then each
// pair of bytes spread into the low bytes of two bf16 lanes of 128.0
__device__ __forceinline__ uint4 word_minus_z(uint32_t w, uint32_t zz) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu, m = 0x43434343u;
    const uint32_t u0 = __byte_perm(lo, hi, 0x5140), u1 = __byte_perm(lo, hi, 0x7362);   // c0..c3, c4..c7
    return make_uint4(bf2_sub(__byte_perm(u0, m, 0x4140), zz), bf2_sub(__byte_perm(u0, m, 0x4342), zz),
                      bf2_sub(__byte_perm(u1, m, 0x4140), zz), bf2_sub(__byte_perm(u1, m, 0x4342), zz));
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
// every thread of the role waits on (and arrives at) the barrier itself:
// measured faster here than one elected lane per warp
__device__ __forceinline__ bool role_wait(uint64_t *bar, uint32_t parity, uint32_t limit, const int *timeout) {
    return *reinterpret_cast<const volatile int *>(timeout) == 0 && umma::mbar_wait(bar, parity, limit);
}
__device__ __forceinline__ void role_arrive(uint64_t *bar) { umma::mbar_arrive(bar); }

__device__ __forceinline__ uint64_t f2(float a, float b) {
    return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

template <int BN>
struct Ctl {
    uint64_t afull[kSA], aempty[kSA];                         // A buffers: converted / read by the MMAs
    uint64_t bfull[4], bempty[4];                             // activation stages: landed / read
    uint64_t accf[2], acce[2];
    uint64_t cfull[ring_boxes<BN>()], cempty[ring_boxes<BN>()];                         // code boxes landed / read by every converter
    uint64_t drain[2];                 // after a timeout: each issuer's MMAs in flight have finished
    uint64_t never;                    // nothing arrives here (the stall test)
    uint32_t tmem;
    int timeout;
    int drained;                       // 0 after a drain that ran out
};

template <int BN>
constexpr size_t smem_total() {
    return (size_t)n_stages<BN>() * stage_bytes<BN>() + (size_t)ring_boxes<BN>() * kCodeBox + sizeof(Ctl<BN>) + 1024;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_umma_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                      const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y, int ldy,
                      int32_t *st, int C, uint32_t wait_limit, int stall, KvOut kv) {
    constexpr int S = n_stages<BN>();
    constexpr int kStage = stage_bytes<BN>();
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 128, "token tile");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // stages 1024-aligned (the swizzle pattern is a function of the address)
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int SC = ring_boxes<BN>();
    uint8_t *codes = stages + (size_t)S * kStage;                 // SC boxes of kCodeBox bytes
    Ctl<BN> &sm = *reinterpret_cast<Ctl<BN> *>(codes + (size_t)SC * kCodeBox);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // cluster of C CTAs splits the groups of one 128-channel tile
    const int rank = C > 1 ? (int)umma::cluster_rank() : 0;
    const int n0 = (blockIdx.x / C) * kTileN, t0 = blockIdx.y * BN;
    const int G = K / kGroup;
    const int g_lo = (int)(((long long)rank * G) / C), g_hi = (int)(((long long)(rank + 1) * G) / C);
    const int NG = g_hi - g_lo;                          // this CTA's groups
    // TMEM: two accumulators of kBuf columns, then kSA A buffers of 64
    constexpr uint32_t kBuf = BN <= 32 ? 32 : BN <= 64 ? 64 : 128;
    constexpr uint32_t kAcol = 2 * kBuf;
    constexpr uint32_t kCols = kAcol + 64 * kSA <= 256 ? 256 : 512;

    if (warp == 0) umma::tmem_alloc(&sm.tmem, kCols);
    if (tid == 0) {
        for (int s = 0; s < kSA; ++s) {
            umma::mbar_init(&sm.afull[s], kConv);
            umma::mbar_init(&sm.aempty[s], 1);
        }
        for (int s = 0; s < S; ++s) {
            umma::mbar_init(&sm.bfull[s], 1);
            umma::mbar_init(&sm.bempty[s], 1);
        }
        for (int c = 0; c < SC; ++c) {
            umma::mbar_init(&sm.cfull[c], 1);
            umma::mbar_init(&sm.cempty[c], kConv);
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(&sm.accf[b], 1);
            umma::mbar_init(&sm.acce[b], kEpilogue);
        }
        umma::mbar_init(&sm.drain[0], 1);
        umma::mbar_init(&sm.drain[1], 1);
        umma::mbar_init(&sm.never, 1);
        sm.timeout = 0;
        sm.drained = 1;
        umma::mbar_fence_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        umma::prefetch_tmap(&tx);
        umma::prefetch_tmap(&tw);
    }
    pdl_launch_dependents();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    bool issued = false;                          // MMAs issued (MMA lane 0)
    int copies = 0;                               // activation stages issued (copy lane 1) / code boxes (lane 0)
    auto timed_out = [&]() { return *reinterpret_cast<volatile int *>(&sm.timeout) != 0; };
    // epilogue partial sums: per thread (row n, token half) BN / 2 values
    constexpr int kHalf = BN / 2;
    uint64_t acc[kHalf / 2];
    bool epi_ok = false;

    if (warp < kConv / 32) {
        // ------------------------------------------------------ weight converters
        // warp w: channels r = 32 (w % 4) + lane (its TMEM lanes), k half
        // h = w / 4 of each group; the thread's 32 code bytes of a group come
        // from the code box (row r, 16-byte chunks 4 (l % 2) + 2 h + {0, 1},
        // 128-byte swizzle); the zero points kD groups ahead in registers
        constexpr int kD = 8;
        const int r = 32 * (warp & 3) + lane, h = warp >> 2, n = n0 + r;
        const bool row_ok = n < N;
        const uint32_t *zrow = sz + (size_t)(row_ok ? n : 0) * G;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t zring[kD];
#pragma unroll
        for (int p = 0; p < kD; ++p) zring[p] = (row_ok && p < NG) ? __ldg(zrow + g_lo + p) : 0u;
        bool ok = true;
        for (int lb = 0; lb < NG && ok; lb += kD) {
#pragma unroll
            for (int p = 0; p < kD; ++p) {
                const int l = lb + p;
                if (l >= NG) break;
                const int sa = l % kSA, c = (l >> 1) % SC;
                // this group's codes (the box holds groups 2 (l / 2), + 1)
                if ((l & 1) == 0 && !role_wait(&sm.cfull[c], ((l >> 1) / SC) & 1, wait_limit, &sm.timeout)) {
                    atomicExch(&sm.timeout, 1);
                    ok = false;
                    break;
                }
                const uint8_t *crow = codes + (size_t)c * kCodeBox + (size_t)r * kAtom;
                const int j0 = 4 * (l & 1) + 2 * h;
                const uint4 c0 = *reinterpret_cast<const uint4 *>(crow + ((j0 ^ (r & 7)) << 4));
                const uint4 c1 = *reinterpret_cast<const uint4 *>(crow + (((j0 + 1) ^ (r & 7)) << 4));
                // the box's next contents come by TMA (the async proxy): these
                // reads are fenced against it before the box is released
                if ((l & 1) == 1 || l + 1 == NG) {
                    umma::fence_proxy_async();
                    role_arrive(&sm.cempty[c]);
                }
                const uint32_t szc = zring[p];
                if (row_ok && l + kD < NG) zring[p] = __ldg(zrow + g_lo + l + kD);
                const uint32_t zb =
                    float_to_bf16_bits(128.0f + __half2float(__ushort_as_half((uint16_t)(szc >> 16))));
                const uint32_t zz = zb | (zb << 16);
                // 64 codes of row r (k = 64 h ..) -> 32 bf16 pairs
                const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 q = word_minus_z(words[j], zz);   // rows past N: zero codes, z = 0 -> 0
                    v[4 * j] = q.x;
                    v[4 * j + 1] = q.y;
                    v[4 * j + 2] = q.z;
                    v[4 * j + 3] = q.w;
                }
                // A buffer sa is free once the MMAs of group l - kSA have read it
                if (l >= kSA && !role_wait(&sm.aempty[sa], ((l / kSA) - 1) & 1, wait_limit, &sm.timeout)) {
                    atomicExch(&sm.timeout, 1);
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                umma::tmem_st32(tmem + lane_off + kAcol + (uint32_t)(sa * 64 + h * 32), v);
                umma::tmem_st_wait();
                umma::fence_before_sync();
                role_arrive(&sm.afull[sa]);
            }
        }
    } else if (warp < kMmaWarp) {
        // ------------------------------------------------------------ epilogue
        pdl_wait();
        constexpr int kW = kHalf % 16 == 0 ? 16 : 8;
        const int eq = warp & 3, eh = (warp - kConv / 32) >> 2;
        const int n = n0 + eq * 32 + lane;
        const bool row_ok = n < N;
#pragma unroll
        for (int i = 0; i < kHalf / 2; ++i) acc[i] = 0;
        bool ok = true;
        uint32_t szn = row_ok && NG > 0 ? __ldg(sz + (size_t)n * G + g_lo) : 0u;
        for (int l = 0; l < NG && ok; ++l) {
            const int buf = l & 1;
            const uint32_t szw = szn;
            if (row_ok && l + 1 < NG) szn = __ldg(sz + (size_t)n * G + g_lo + l + 1);
            const float sn = __half2float(__ushort_as_half((uint16_t)(szw & 0xFFFF)));
            const uint64_t s2 = f2(sn, sn);
            if (!role_wait(&sm.accf[buf], (l >> 1) & 1, wait_limit, &sm.timeout)) {
                atomicExch(&sm.timeout, 1);
                ok = false;
                break;
            }
            umma::fence_after_sync();
#pragma unroll
            for (int c0 = 0; c0 < kHalf; c0 += kW) {
                uint32_t v[kW];
                const uint32_t ta = tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(buf * kBuf + eh * kHalf + c0);
                umma::tmem_ld_cols<kW>(ta, *reinterpret_cast<uint32_t(*)[kW]>(v));
                umma::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < kW; j += 2)
                    acc[(c0 + j) / 2] = fma2(f2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c0 + j) / 2]);
            }
            umma::fence_before_sync();
            role_arrive(&sm.acce[buf]);
        }
        epi_ok = ok;
        if (C == 1 && ok && row_ok) {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
                const int m = t0 + eh * kHalf + 2 * i;
                if (m < M) {
                    const uint16_t v16 = float_to_bf16_bits(__uint_as_float((uint32_t)acc[i]));
                    y[(size_t)m * ldy + n] = v16;
                    kv_store(kv, m, n, v16);
                }
                if (m + 1 < M) {
                    const uint16_t v16 = float_to_bf16_bits(__uint_as_float((uint32_t)(acc[i] >> 32)));
                    y[(size_t)(m + 1) * ldy + n] = v16;
                    kv_store(kv, m + 1, n, v16);
                }
            }
        }
    } else if (warp < kTmaWarp) {
        // ------------------------------------------------------------ MMA issuers
        // issuer i takes groups l = i, i + 2, ...: accumulator i, A buffers
        // and activation stages of parity i (kSA and S are even), so each
        // barrier it polls is at most one phase ahead of the last it saw
        const int iss = warp - kMmaWarp;
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(1, 1, kTileN, BN);
            if (stall && iss == 0 && !umma::mbar_wait(&sm.never, 0, wait_limit)) atomicExch(&sm.timeout, 1);
            for (int l = iss; l < NG; l += 2) {
                const int sa = l % kSA, sb = l % S, buf = l & 1;
                if (timed_out() || !umma::mbar_wait(&sm.afull[sa], (l / kSA) & 1, wait_limit) ||
                    !umma::mbar_wait(&sm.bfull[sb], (l / S) & 1, wait_limit) ||
                    (l >= 2 && !umma::mbar_wait(&sm.acce[buf], ((l >> 1) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    break;
                }
                umma::fence_after_sync();
                const uint32_t b0 = umma::smem_addr(stages + (size_t)sb * kStage);
                const uint32_t a0 = tmem + kAcol + (uint32_t)(sa * 64);
                const uint32_t d = tmem + (uint32_t)(buf * kBuf);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {               // K = 16 bf16: 8 TMEM columns of A, 32 bytes of B
                    const uint64_t db = desc_sw128(b0 + (kk >> 2) * BN * kAtom);
                    umma::mma_bf16_ta(d, a0 + 8 * kk, db + 2 * (kk & 3), idesc, kk != 0 ? 1u : 0u);
                }
                umma::mma_commit(&sm.aempty[sa]);
                umma::mma_commit(&sm.bempty[sb]);
                umma::mma_commit(&sm.accf[buf]);
                issued = true;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ copies
        const int NP = (NG + 1) / 2;                      // code boxes: two groups each
        if (lane == 0) {
            // code boxes: the first SC before the dependency wait
            for (int p = 0; p < NP; ++p) {
                const int c = p % SC;
                if (p >= SC && (timed_out() || !umma::mbar_wait(&sm.cempty[c], ((p / SC) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    break;
                }
                umma::mbar_arrive_expect_tx(&sm.cfull[c], (uint32_t)kCodeBox);
                umma::tma_load_2d(codes + (size_t)c * kCodeBox, &tw, (g_lo + 2 * p) * (kGroup / 2), n0, &sm.cfull[c]);
                copies = p + 1;
            }
        } else if (lane == 1) {
            pdl_wait();
            for (int l = 0; l < NG; ++l) {
                const int s = l % S, g = g_lo + l;
                if (l >= S && (timed_out() || !umma::mbar_wait(&sm.bempty[s], ((l / S) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    break;
                }
                uint8_t *b = stages + (size_t)s * kStage;
                umma::mbar_arrive_expect_tx(&sm.bfull[s], (uint32_t)(BN * 2 * kAtom));
                umma::tma_load_2d(b, &tx, g * 2 * kAtom, t0, &sm.bfull[s]);
                umma::tma_load_2d(b + BN * kAtom, &tx, g * 2 * kAtom + kAtom, t0, &sm.bfull[s]);
                copies = l + 1;
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
            for (int p = std::max(0, copies - SC); p < copies; ++p)
                if (!umma::mbar_wait(&sm.cfull[p % SC], (p / SC) & 1, kWaitLimit)) sm.drained = 0;
        if (warp == kTmaWarp && lane == 1)
            for (int l = std::max(0, copies - S); l < copies; ++l)
                if (!umma::mbar_wait(&sm.bfull[l % S], (l / S) & 1, kWaitLimit)) sm.drained = 0;
        if (warp >= kMmaWarp && warp < kTmaWarp && lane == 0 && issued) {
            umma::mma_commit(&sm.drain[warp - kMmaWarp]);
            if (!umma::mbar_wait(&sm.drain[warp - kMmaWarp], 0, kWaitLimit)) sm.drained = 0;
        }
        __syncthreads();
    }
    if (C > 1) {
        // split groups: every CTA's partials -> its shared memory (the operand
        // stages are free now: all copies and MMAs have completed); rank 0
        // adds them in rank order and stores bf16
        float *red = reinterpret_cast<float *>(stages);            // [BN tokens][128 channels]
        const int eq = warp & 3, eh = (warp - kConv / 32) >> 2, row = eq * 32 + lane;
        const bool epi_warp = warp >= kConv / 32 && warp < kMmaWarp;
        const bool reuse = sm.drained != 0;                        // the operand stages are free
        if (epi_warp && reuse) {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
                const int t = eh * kHalf + 2 * i;
                red[(size_t)t * kTileN + row] = epi_ok ? __uint_as_float((uint32_t)acc[i]) : 0.0f;
                red[(size_t)(t + 1) * kTileN + row] = epi_ok ? __uint_as_float((uint32_t)(acc[i] >> 32)) : 0.0f;
            }
        }
        umma::cluster_sync();
        if (rank == 0 && epi_warp && reuse && !sm.timeout) {
            const int n = n0 + row;
            if (n < N) {
                for (int t = eh * kHalf; t < eh * kHalf + kHalf; ++t) {
                    const int m = t0 + t;
                    if (m >= M) break;
                    float sum = red[(size_t)t * kTileN + row];
                    for (int q = 1; q < C; ++q) sum += umma::ld_peer_f32(&red[(size_t)t * kTileN + row], (uint32_t)q);
                    const uint16_t v16 = float_to_bf16_bits(sum);
                    y[(size_t)m * ldy + n] = v16;
                    kv_store(kv, m, n, v16);
                }
            }
        }
        umma::cluster_sync();
    }
    if (tid == 0 && sm.timeout) flag(st, QSPEC_ERR_TIMEOUT);
    if (warp == 0) umma::tmem_free(tmem, kCols);
}

template <int BN>
int launch_bn(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
              uint16_t *y, int ldy, int32_t *st, cudaStream_t stream, uint32_t wait_limit, int stall,
              const KvOut &kv) {
    static_assert(sizeof(float) * BN * kTileN <= (size_t)n_stages<BN>() * stage_bytes<BN>(),
                  "partials fit in the operand stages");
    CUtensorMap tx, tw;
    // the activations as bytes: rows of K bf16, boxes of 128 bytes x BN tokens;
    // the packed codes: rows of K / 2 bytes, boxes of 128 bytes x 128 channels
    if (byte_tmap_sw128(&tx, x, M, 2 * K, (size_t)ldx * 2, BN) ||
        byte_tmap_sw128(&tw, packed, N, K / 2, (size_t)K / 2, kTileN))
        return QSPEC_ERR_UNSUPPORTED;
    const size_t smem = smem_total<BN>();
    int rc = smem_limit_once(reinterpret_cast<const void *>(&w4a16_umma_kernel<BN>), (int)smem);
    if (rc) return rc;
    const int n_tiles = (N + kTileN - 1) / kTileN, token_tiles = (M + BN - 1) / BN, G = K / kGroup;
    // split the groups over a cluster (2, 4 or 8 CTAs: sizes that pack into
    // the GPCs) when the tiles alone leave SMs idle
    int C = 1;
    while (C < 8 && n_tiles * token_tiles * C * 2 <= sm_count() && 2 * C * 2 <= G) C *= 2;
    dim3 grid((unsigned)(n_tiles * C), (unsigned)token_tiles);
    if (C == 1)
        return launch_pdl("qspec_linear_w4a16", w4a16_umma_kernel<BN>, grid, dim3(kThreads), smem, stream, tx, tw,
                          sz, M, N, K, y, ldy, st, C, wait_limit, stall, kv);
    return launch_pdl_cluster("qspec_linear_w4a16", w4a16_umma_kernel<BN>, grid, dim3(kThreads), smem, stream, C, tx,
                              tw, sz, M, N, K, y, ldy, st, C, wait_limit, stall, kv);
}

}  // namespace

// Large-M W4A16: ceil(M / 128) token tiles of BN tokens (a multiple of 16,
// 32 ... 128).
int launch_w4a16_tc(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                    uint16_t *y, int ldy, int32_t *st, cudaStream_t stream, uint32_t wait_limit, int stall,
                    const KvOut &kv) {
    const int tiles = (M + 127) / 128, per = (M + tiles - 1) / tiles, bn = std::max(32, (per + 15) / 16 * 16);
    switch (bn) {
        case 32: return launch_bn<32>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        case 48: return launch_bn<48>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        case 64: return launch_bn<64>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        case 80: return launch_bn<80>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        case 96: return launch_bn<96>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        case 112: return launch_bn<112>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
        default: return launch_bn<128>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
    }
}

}  // namespace qspec
