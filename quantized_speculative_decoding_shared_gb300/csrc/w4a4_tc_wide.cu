// w4a4_tc_wide.cu -- a3, W4A4 linear on the Blackwell tensor cores for
// prefill-sized M (256 tokens and more: 128-token tiles).  Measured against
// the decode-batch kernel in w4a4_tc.cu at M = 4096 through Llama-3-8B
// gate/up and down: 275 vs 180 TOPS -- there the epilogue's exact fold, not
// the weight stream, bounds the kernel, and this design's 416 threads leave
// the epilogue 152 registers where the decode-batch kernel's 608 leave 96.
//
// QSPEC summary page, background terms: 4-bit activations times 4-bit
// weights, products accumulated exactly (INT32 in the pages' wording), then
// scaled to 16 bits.  Bit-exact definition (the same as the small-M kernel
// and the CPU oracle):
//   I[m][n][g] = sum_{k in g} q (W - z) ; acc = fmaf((float) I, sx * s, acc)
//   for g ascending from acc = 0 ; y = bf16_rn(acc).
//
// sm_103a has no integer tcgen05 MMA, so the products run as
// tcgen05.mma kind::f8f6f4 with E4M3 operands that hold the integers exactly:
// codes 0..15 (weights, A operand, 128 output channels per CTA) and
// q in [-8, 7] (activations, B operand, BN tokens per CTA).  One K step is
// one 128-wide group (4 MMAs of K = 32).  Every product is an integer of
// magnitude <= 120 and every partial sum of a group stays below 2^14, so the
// fp32 accumulator in TMEM holds sum q W exactly; the epilogue forms
// I = sum q W - z qs exactly in fp32 (|I| <= 13440) and folds it.
//
//   warps 0-3  producers: nibbles -> E4M3 bytes (byte permutes), written to
//              shared memory in the no-swizzle K-major core-matrix layout,
//              with the tokens' sx / qs of the group
//   warps 4-11 epilogue, two warpgroups on the same TMEM lanes, each with half
//              of the token columns: per group, TMEM -> registers, I and the
//              ordered fp32 fold in registers (packed f32x2); finally bf16
//   warp 12    issues the MMAs into one of two TMEM accumulators per group
// Bounded waits everywhere (the limit is a kernel argument; a test can also
// make the MMA issuer wait on a barrier nothing arrives at).  After a
// timeout (QSPEC_ERR_TIMEOUT) every role leaves its loop -- the epilogue
// warpgroups together, through a barrier that ORs their failure flags, since
// they also meet at a named barrier -- the MMAs issued are drained with a
// bounded wait, and the tensor memory is freed (even if the drain itself ran
// out: the next kernel on the SM would otherwise wait for it without bound).
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

namespace wide {

constexpr int kStages = 4;
constexpr int kTileN = 128;        // output channels per CTA (MMA M)
constexpr int kKB = kGroup;        // bytes of K per row per stage (E4M3)
constexpr int kProducers = 128;
constexpr int kEpilogue = 256;        // two warpgroups, each folds half of the token columns
constexpr int kThreads = kProducers + kEpilogue + 32;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// E4M3 bytes of the unsigned codes 0..15 in the low 16 bits' nibbles of `w`.
// prmt's selector nibble bit 3 replicates the sign bit of the chosen byte; all
// table bytes are positive, so codes >= 8 give 0 from the first lookup and
// codes < 8 give 0 from the second (which looks up ~w).
__device__ __forceinline__ uint32_t e4m3_codes4(uint32_t w, uint32_t nw) {
    const uint32_t t0 = 0x44403800u, t1 = 0x4E4C4A48u;   // E4M3 of 0..7
    const uint32_t u0 = 0x54555657u, u1 = 0x50515253u;   // E4M3 of 15..8 (index 7 - (c - 8))
    return prmt(t0, t1, w) | prmt(u0, u1, nw);
}

// eight codes (one word) -> two words of E4M3 bytes in k order
__device__ __forceinline__ uint2 e4m3_codes8(uint32_t w) {
    const uint32_t nw = ~w;
    return make_uint2(e4m3_codes4(w, nw), e4m3_codes4(w >> 16, nw >> 16));
}

// eight two's-complement nibbles q in [-8, 7] -> two words of E4M3 bytes:
// magnitude through the code tables, sign bit set from the nibble's bit 3
__device__ __forceinline__ uint2 e4m3_acts8(uint32_t w) {
    const uint32_t s4 = (w >> 3) & 0x11111111u;            // sign of each nibble
    const uint32_t mag = (w ^ (s4 * 15u)) + s4;            // |q| per nibble, 0..8, no carries
    const uint32_t nmag = ~mag;
    const uint32_t k80 = 0x80808080u;
    // byte i of prmt(k80, k80, w) is 0xFF when nibble i is negative, else 0x80
    const uint32_t sg_lo = (prmt(k80, k80, w) << 7) & 0x80808080u;
    const uint32_t sg_hi = (prmt(k80, k80, w >> 16) << 7) & 0x80808080u;
    return make_uint2(e4m3_codes4(mag, nmag) | sg_lo, e4m3_codes4(mag >> 16, nmag >> 16) | sg_hi);
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

template <int BN>
struct Smem {
    uint8_t a[kStages][kTileN * kKB];
    uint8_t b[kStages][BN * kKB];
    float esx[2][BN];                  // epilogue-owned: sx of the group's tokens
    float enqs[2][BN];                 // -qs as float (exact)
    uint64_t full[kStages], empty[kStages], accf[2], acce[2];
    uint64_t drain;                    // after a timeout: the MMAs in flight have finished
    uint64_t never;                    // nothing arrives here (the stall test)
    uint32_t tmem;
    int timeout;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_umma_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ sx, const int32_t *__restrict__ qs,
                     const uint8_t *__restrict__ packed, const uint32_t *__restrict__ sz, int M, int N, int K,
                     uint16_t *__restrict__ y, int ldy, int32_t *__restrict__ dbg_I, int32_t *st,
                     uint32_t wait_limit, int stall) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem<BN> &sm = *reinterpret_cast<Smem<BN> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kTileN, t0 = blockIdx.y * BN;
    const int G = K / kGroup;
    constexpr uint32_t kCols = 2 * (BN <= 32 ? 32 : BN <= 64 ? 64 : 128);
    constexpr uint32_t kBuf = kCols / 2;

    if (warp == 0) umma::tmem_alloc(&sm.tmem, kCols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            umma::mbar_init(&sm.full[s], kProducers);
            umma::mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(&sm.accf[b], 1);
            umma::mbar_init(&sm.acce[b], kEpilogue);
        }
        umma::mbar_init(&sm.drain, 1);
        umma::mbar_init(&sm.never, 1);
        sm.timeout = 0;
        umma::mbar_fence_init();
    }
    pdl_launch_dependents();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    bool issued = false;                          // MMAs issued (MMA lane 0)
    auto timed_out = [&]() { return *reinterpret_cast<volatile int *>(&sm.timeout) != 0; };

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        const int r = tid, n = n0 + r;
        const bool row_ok = n < N;
        const uint4 *wrow = reinterpret_cast<const uint4 *>(packed + (size_t)(row_ok ? n : 0) * (K / 2));
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = row_ok ? __ldg(wrow + u) : make_uint4(0, 0, 0, 0);
        pdl_wait();
        for (int g = 0; g < G; ++g) {
            const int s = g % kStages;
            if (g >= kStages &&
                (timed_out() || !umma::mbar_wait(&sm.empty[s], ((g / kStages) - 1) & 1, wait_limit))) {
                atomicExch(&sm.timeout, 1);
                break;
            }
            uint4 cw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) cw[u] = w[u];
            if (row_ok && g + 1 < G) {
#pragma unroll
                for (int u = 0; u < 4; ++u) w[u] = __ldg(wrow + (g + 1) * 4 + u);
            }
            // weights: 128 codes of row r -> 8 chunks of 16 E4M3 bytes
            uint8_t *a = sm.a[s];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint2 e0 = e4m3_codes8(cw[u].x), e1 = e4m3_codes8(cw[u].y);
                const uint2 e2 = e4m3_codes8(cw[u].z), e3 = e4m3_codes8(cw[u].w);
                *reinterpret_cast<uint4 *>(a + umma::core_offset(r, 2 * u, kKB)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
                *reinterpret_cast<uint4 *>(a + umma::core_offset(r, 2 * u + 1, kKB)) =
                    make_uint4(e2.x, e2.y, e3.x, e3.y);
            }
            // activations: BN tokens x 64 bytes of nibbles -> BN x 128 E4M3 bytes
            uint8_t *b = sm.b[s];
            for (int c = tid; c < BN * 4; c += kProducers) {
                const int t = c >> 2, u = c & 3, m = t0 + t;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (m < M) v = __ldg(reinterpret_cast<const uint4 *>(xq + (size_t)m * (K / 2) + (size_t)g * 64) + u);
                const uint2 e0 = e4m3_acts8(v.x), e1 = e4m3_acts8(v.y), e2 = e4m3_acts8(v.z), e3 = e4m3_acts8(v.w);
                *reinterpret_cast<uint4 *>(b + umma::core_offset(t, 2 * u, kKB)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
                *reinterpret_cast<uint4 *>(b + umma::core_offset(t, 2 * u + 1, kKB)) =
                    make_uint4(e2.x, e2.y, e3.x, e3.y);
            }
            umma::fence_proxy_async();
            umma::mbar_arrive(&sm.full[s]);
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ epilogue
        pdl_wait();
        constexpr int kHalf = BN / 2;                 // token columns per warpgroup
        const int eq = warp & 3;                      // TMEM lanes 32 eq .. 32 eq + 31
        const int eh = (warp - 4) >> 2;               // column half
        const int et = tid - kProducers;              // 0 .. 255
        const int n = n0 + eq * 32 + lane;
        const bool row_ok = n < N;
        uint64_t acc[kHalf / 2];
#pragma unroll
        for (int i = 0; i < kHalf / 2; ++i) acc[i] = 0;
        bool ok = true;
        for (int g = 0; g < G; ++g) {
            const int buf = g & 1;
            // the group's token scales into the epilogue's own double buffer; the
            // barrier also orders this write after every epilogue thread's reads
            // of the same buffer two groups ago, and tells every epilogue thread
            // whether any of them has given up (all leave together)
            for (int t = et; t < BN; t += kEpilogue) {
                const int m = t0 + t;
                sm.esx[buf][t] = m < M ? sx[(size_t)m * G + g] : 0.0f;
                sm.enqs[buf][t] = m < M ? -(float)qs[(size_t)m * G + g] : 0.0f;
            }
            uint32_t any_failed;
            asm volatile(
                "{.reg .pred p, q; setp.eq.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q;}\n"
                : "=r"(any_failed)
                : "r"(ok ? 1u : 0u), "r"(kEpilogue)
                : "memory");
            if (any_failed) break;
            if (timed_out() || !umma::mbar_wait(&sm.accf[buf], (g >> 1) & 1, wait_limit)) {
                atomicExch(&sm.timeout, 1);
                ok = false;
                continue;                             // to the barrier, where all leave
            }
            umma::fence_after_sync();
            const uint32_t szw = row_ok ? __ldg(sz + (size_t)n * G + g) : 0u;
            const float sn = __half2float(__ushort_as_half((uint16_t)(szw & 0xFFFF)));
            const float zn = __half2float(__ushort_as_half((uint16_t)(szw >> 16)));
            const uint64_t s2 = f2(sn, sn), z2 = f2(zn, zn);
#pragma unroll
            for (int c0 = 0; c0 < kHalf; c0 += (kHalf < 32 ? kHalf : 32)) {
                constexpr int kW = kHalf < 32 ? kHalf : 32;
                uint32_t v[32];
                const uint32_t ta = tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(buf * kBuf + eh * kHalf + c0);
                if (kW == 32)
                    umma::tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(v));
                else
                    umma::tmem_ld16(ta, v);
                umma::tmem_ld_wait();
                // no branch inside the plain loop, so the pairs' loads and
                // packed operations interleave; the debug output takes its own
                if (dbg_I == nullptr) {
#pragma unroll
                    for (int j = 0; j < kW; j += 2) {
                        const int t = eh * kHalf + c0 + j;
                        // I = sum qW - z qs (exact), c = sx * s, acc = fma(I, c, acc)
                        const uint64_t nqs2 = *reinterpret_cast<const uint64_t *>(&sm.enqs[buf][t]);
                        const uint64_t sx2 = *reinterpret_cast<const uint64_t *>(&sm.esx[buf][t]);
                        const uint64_t I2 = fma2(z2, nqs2, f2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])));
                        acc[(c0 + j) / 2] = fma2(I2, mul2(sx2, s2), acc[(c0 + j) / 2]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kW; j += 2) {
                        const int t = eh * kHalf + c0 + j;
                        const uint64_t nqs2 = *reinterpret_cast<const uint64_t *>(&sm.enqs[buf][t]);
                        const uint64_t sx2 = *reinterpret_cast<const uint64_t *>(&sm.esx[buf][t]);
                        const uint64_t I2 = fma2(z2, nqs2, f2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])));
                        acc[(c0 + j) / 2] = fma2(I2, mul2(sx2, s2), acc[(c0 + j) / 2]);
                        if (row_ok) {
                            const int m0 = t0 + t;
                            if (m0 < M) dbg_I[((size_t)m0 * N + n) * G + g] = (int32_t)__uint_as_float((uint32_t)I2);
                            if (m0 + 1 < M)
                                dbg_I[((size_t)(m0 + 1) * N + n) * G + g] =
                                    (int32_t)__uint_as_float((uint32_t)(I2 >> 32));
                        }
                    }
                }
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.acce[buf]);
        }
        if (ok && row_ok) {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
                const int m = t0 + eh * kHalf + 2 * i;
                if (m < M) y[(size_t)m * ldy + n] = float_to_bf16_bits(__uint_as_float((uint32_t)acc[i]));
                if (m + 1 < M) y[(size_t)(m + 1) * ldy + n] = float_to_bf16_bits(__uint_as_float((uint32_t)(acc[i] >> 32)));
            }
        }
    } else {
        // ------------------------------------------------------------ MMA issuer
        pdl_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(0, 0, kTileN, BN);
            if (stall && !umma::mbar_wait(&sm.never, 0, wait_limit)) atomicExch(&sm.timeout, 1);
            for (int g = 0; g < G; ++g) {
                const int s = g % kStages, buf = g & 1;
                if (timed_out() || !umma::mbar_wait(&sm.full[s], (g / kStages) & 1, wait_limit) ||
                    (g >= 2 && !umma::mbar_wait(&sm.acce[buf], ((g >> 1) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    break;
                }
                umma::fence_after_sync();
                const uint32_t a0 = umma::smem_addr(sm.a[s]), b0 = umma::smem_addr(sm.b[s]);
                const uint32_t d = tmem + (uint32_t)(buf * kBuf);
#pragma unroll
                for (int j = 0; j < kKB / 32; ++j) {       // K = 32 E4M3 = 2 core matrices per MMA
                    const uint64_t da = umma::smem_desc(a0 + j * 256, 128, (kKB / 16) * 128);
                    const uint64_t db = umma::smem_desc(b0 + j * 256, 128, (kKB / 16) * 128);
                    umma::mma_e4m3(d, da, db, idesc, j != 0);
                }
                umma::mma_commit(&sm.empty[s]);
                umma::mma_commit(&sm.accf[buf]);
                issued = true;
            }
        }
        __syncwarp();
    }
    umma::fence_before_sync();
    __syncthreads();
    // after a timeout, the MMAs already issued finish (bounded wait) before
    // the TMEM they write is freed; sm.timeout is settled at this barrier
    if (sm.timeout) {
        if (warp == kThreads / 32 - 1 && lane == 0 && issued) {
            umma::mma_commit(&sm.drain);
            umma::mbar_wait(&sm.drain, 0, kWaitLimit);
        }
        __syncthreads();
    }
    if (tid == 0 && sm.timeout) flag(st, QSPEC_ERR_TIMEOUT);
    if (warp == 0) umma::tmem_free(tmem, kCols);
}

template <int BN>
int launch_bn(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed, const uint32_t *sz,
              int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st, cudaStream_t stream,
              uint32_t wait_limit, int stall) {
    const size_t smem = sizeof(Smem<BN>) + 1024;
    int rc = smem_limit_once(reinterpret_cast<const void *>(&w4a4_umma_kernel<BN>), (int)smem);
    if (rc) return rc;
    dim3 grid((unsigned)((N + kTileN - 1) / kTileN), (unsigned)((M + BN - 1) / BN));
    return launch_pdl("qspec_linear_w4a4", w4a4_umma_kernel<BN>, grid, dim3(kThreads), smem, stream, xq, sx, qs,
                      packed, sz, M, N, K, y, ldy, dbg_I, st, wait_limit, stall);
}

}  // namespace wide

}  // namespace

// Prefill-sized W4A4 on the tensor cores: token tiles of 128.
int launch_w4a4_tc_wide(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                        const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st,
                        cudaStream_t stream, uint32_t wait_limit, int stall) {
    return wide::launch_bn<128>(xq, sx, qs, packed, sz, M, N, K, y, ldy, dbg_I, st, stream, wait_limit, stall);
}

}  // namespace qspec
