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
// One CTA computes a 128 (output channels) x BN (tokens) tile of Y^T:
//   warps 0-3  producers: per group, the packed codes of one channel each ->
//              bf16 (c - z) (the code OR-ed into the mantissa of 128.0 gives
//              128 + c exactly, then an exact subtraction of 128 + z), and
//              the activation rows; both in shared memory in the no-swizzle
//              K-major core-matrix layout, with k permuted within each 8-wide
//              chunk identically on both operands (a dot product does not
//              depend on the order of k)
//   warps 4-11 epilogue, two warpgroups on the same TMEM lanes, each with half
//              of the token columns: per group, TMEM -> registers,
//              y = fma(D, s, y) in packed f32x2; finally bf16
//   warp 12    issues 8 MMAs (K = 16) per group into one of two TMEM buffers
// When the 128-channel tiles alone would leave SMs idle, a cluster of up to 8
// CTAs splits a tile's groups; each CTA keeps its fp32 partial sums, and
// rank 0 reads its peers' partials from distributed shared memory, adds them
// in rank order and stores bf16.
// Bounded waits everywhere (the limit is a kernel argument; a test can also
// make the MMA issuer wait on a barrier nothing arrives at).  After a
// timeout (QSPEC_ERR_TIMEOUT) every role leaves its loop, the MMAs issued are
// drained with a bounded wait, and the tensor memory is freed -- even if the
// drain itself ran out (the next kernel on the SM would otherwise wait for it
// without bound); in that case the split-K reduction, which reuses the
// operand stages the MMAs read, is skipped.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

constexpr int kStages = 3;
constexpr int kTileN = 128;              // output channels per CTA (MMA M)
constexpr int kKB = kGroup * 2;          // bytes of K per row per stage (bf16)
constexpr int kProducers = 128;
constexpr int kEpilogue = 256;
constexpr int kThreads = kProducers + kEpilogue + 32;

__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// eight codes of a word -> bf16 (c - z) in the order k0,k4,k1,k5,k2,k6,k3,k7
__device__ __forceinline__ uint4 codes_minus_z(uint32_t w, uint32_t zz) {
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;   // bf16 128 + c
    return make_uint4(bf2_sub((w & mask) | magic, zz), bf2_sub(((w >> 4) & mask) | magic, zz),
                      bf2_sub(((w >> 8) & mask) | magic, zz), bf2_sub(((w >> 12) & mask) | magic, zz));
}

// eight bf16 activations x0..x7 -> the same order
__device__ __forceinline__ uint4 acts_permuted(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                      __byte_perm(v.y, v.w, 0x7632));
}

__device__ __forceinline__ uint64_t f2(float a, float b) {
    return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

template <int BN>
struct Smem {
    uint8_t a[kStages][kTileN * kKB];
    uint8_t b[kStages][BN * kKB];
    uint64_t full[kStages], empty[kStages], accf[2], acce[2];
    uint64_t drain;                    // after a timeout: the MMAs in flight have finished
    uint64_t never;                    // nothing arrives here (the stall test)
    uint32_t tmem;
    int timeout;
    int drained;                       // 0 after a drain that ran out
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_umma_kernel(const uint16_t *__restrict__ x, int ldx, const uint8_t *__restrict__ packed,
                      const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y, int ldy,
                      int32_t *st, int C, uint32_t wait_limit, int stall, KvOut kv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem<BN> &sm = *reinterpret_cast<Smem<BN> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // cluster of C CTAs splits the groups of one 128-channel tile
    const int rank = C > 1 ? (int)umma::cluster_rank() : 0;
    const int n0 = (blockIdx.x / C) * kTileN, t0 = blockIdx.y * BN;
    const int G = K / kGroup;
    const int g_lo = (int)(((long long)rank * G) / C), g_hi = (int)(((long long)(rank + 1) * G) / C);
    const int NG = g_hi - g_lo;                          // this CTA's groups
    constexpr uint32_t kBuf = BN <= 32 ? 32 : BN <= 64 ? 64 : 128;
    constexpr uint32_t kCols = 2 * kBuf;

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
        sm.drained = 1;
        umma::mbar_fence_init();
    }
    pdl_launch_dependents();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    bool issued = false;                          // MMAs issued (MMA lane 0)
    auto timed_out = [&]() { return *reinterpret_cast<volatile int *>(&sm.timeout) != 0; };
    // epilogue partial sums: per thread (row n, token half) BN / 2 values
    constexpr int kHalf = BN / 2;
    uint64_t acc[kHalf / 2];
    bool epi_ok = false;

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        // weights: kD groups in flight per thread (one row each); activations
        // of a group: all of a thread's chunks loaded before any is stored
        constexpr int kD = 2;
        constexpr int kChunks = BN * 16 / kProducers;  // 16-byte activation chunks per thread per group
        const int r = tid, n = n0 + r;
        const bool row_ok = n < N;
        const uint4 *wrow = reinterpret_cast<const uint4 *>(packed + (size_t)(row_ok ? n : 0) * (K / 2));
        uint4 ring[kD][4];
        uint32_t zring[kD];
#pragma unroll
        for (int p = 0; p < kD; ++p) {
            const int g = g_lo + p;
            if (g < g_hi) {
#pragma unroll
                for (int u = 0; u < 4; ++u) ring[p][u] = __ldg(wrow + (size_t)g * 4 + u);
                zring[p] = row_ok ? __ldg(sz + (size_t)n * G + g) : 0u;
            }
        }
        pdl_wait();
        bool ok = true;
        for (int lb = 0; lb < NG && ok; lb += kD) {
#pragma unroll
            for (int p = 0; p < kD; ++p) {
                const int l = lb + p, g = g_lo + l;
                if (l >= NG) break;
                const int s = l % kStages;
                if (l >= kStages &&
                    (timed_out() || !umma::mbar_wait(&sm.empty[s], ((l / kStages) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    ok = false;
                    break;
                }
                uint4 cw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) cw[u] = ring[p][u];
                const uint32_t szc = zring[p];
                if (l + kD < NG) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) ring[p][u] = __ldg(wrow + (size_t)(g + kD) * 4 + u);
                    zring[p] = row_ok ? __ldg(sz + (size_t)n * G + g + kD) : 0u;
                }
                const uint32_t zb =
                    float_to_bf16_bits(128.0f + __half2float(__ushort_as_half((uint16_t)(szc >> 16))));
                const uint32_t zz = zb | (zb << 16);
                // weights: 128 codes of row r -> 16 chunks of 8 bf16
                uint8_t *a = sm.a[s];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t words[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = row_ok ? codes_minus_z(words[q], zz) : make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(a + umma::core_offset(r, 4 * u + q, kKB)) = v;
                    }
                }
                // this group's activation chunks, in batches: loads first
                uint8_t *b = sm.b[s];
                constexpr int kBatch = kChunks % 8 == 0 ? 8 : kChunks % 6 == 0 ? 6 : 4;
                static_assert(kChunks % kBatch == 0, "batches cover the chunks exactly");
#pragma unroll
                for (int j0 = 0; j0 < kChunks; j0 += kBatch) {
                    uint4 av[kBatch];
#pragma unroll
                    for (int j = 0; j < kBatch; ++j) {
                        const int c = tid + (j0 + j) * kProducers, t = c >> 4, jj = c & 15, m = t0 + t;
                        av[j] = m < M ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)m * ldx +
                                                                              (size_t)g * kGroup + jj * 8))
                                      : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int j = 0; j < kBatch; ++j) {
                        const int c = tid + (j0 + j) * kProducers, t = c >> 4, jj = c & 15;
                        *reinterpret_cast<uint4 *>(b + umma::core_offset(t, jj, kKB)) = acts_permuted(av[j]);
                    }
                }
                umma::fence_proxy_async();
                umma::mbar_arrive(&sm.full[s]);
            }
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ epilogue
        pdl_wait();
        constexpr int kW = kHalf % 32 == 0 ? 32 : 16;
        const int eq = warp & 3, eh = (warp - 4) >> 2;
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
            if (timed_out() || !umma::mbar_wait(&sm.accf[buf], (l >> 1) & 1, wait_limit)) {
                atomicExch(&sm.timeout, 1);
                ok = false;
                break;
            }
            umma::fence_after_sync();
#pragma unroll
            for (int c0 = 0; c0 < kHalf; c0 += kW) {
                uint32_t v[32];
                const uint32_t ta = tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(buf * kBuf + eh * kHalf + c0);
                if (kW == 32)
                    umma::tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(v));
                else
                    umma::tmem_ld16(ta, v);
                umma::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < kW; j += 2)
                    acc[(c0 + j) / 2] = fma2(f2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c0 + j) / 2]);
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.acce[buf]);
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
    } else {
        // ------------------------------------------------------------ MMA issuer
        pdl_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(1, 1, kTileN, BN);
            if (stall && !umma::mbar_wait(&sm.never, 0, wait_limit)) atomicExch(&sm.timeout, 1);
            for (int l = 0; l < NG; ++l) {
                const int s = l % kStages, buf = l & 1;
                if (timed_out() || !umma::mbar_wait(&sm.full[s], (l / kStages) & 1, wait_limit) ||
                    (l >= 2 && !umma::mbar_wait(&sm.acce[buf], ((l >> 1) - 1) & 1, wait_limit))) {
                    atomicExch(&sm.timeout, 1);
                    break;
                }
                umma::fence_after_sync();
                const uint32_t a0 = umma::smem_addr(sm.a[s]), b0 = umma::smem_addr(sm.b[s]);
                const uint32_t d = tmem + (uint32_t)(buf * kBuf);
#pragma unroll
                for (int j = 0; j < kKB / 32; ++j) {       // K = 16 bf16 = 2 core matrices per MMA
                    const uint64_t da = umma::smem_desc(a0 + j * 256, 128, (kKB / 16) * 128);
                    const uint64_t db = umma::smem_desc(b0 + j * 256, 128, (kKB / 16) * 128);
                    umma::mma_bf16(d, da, db, idesc, j != 0);
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
            if (!umma::mbar_wait(&sm.drain, 0, kWaitLimit)) sm.drained = 0;
        }
        __syncthreads();
    }
    if (C > 1) {
        // split groups: every CTA's partials -> its shared memory (the operand
        // stages are free now: all MMAs have completed); rank 0 adds them in
        // rank order and stores bf16
        float *red = reinterpret_cast<float *>(smem_raw);          // [BN tokens][128 channels]
        const int eq = warp & 3, eh = (warp - 4) >> 2, row = eq * 32 + lane;
        const bool reuse = sm.drained != 0;                        // the operand stages are free
        if (warp >= 4 && warp < 12 && reuse) {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
                const int t = eh * kHalf + 2 * i;
                red[(size_t)t * kTileN + row] = epi_ok ? __uint_as_float((uint32_t)acc[i]) : 0.0f;
                red[(size_t)(t + 1) * kTileN + row] = epi_ok ? __uint_as_float((uint32_t)(acc[i] >> 32)) : 0.0f;
            }
        }
        umma::cluster_sync();
        if (rank == 0 && warp >= 4 && warp < 12 && reuse && !sm.timeout) {
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
    static_assert(sizeof(float) * BN * kTileN <= sizeof(Smem<BN>::a) + sizeof(Smem<BN>::b),
                  "partials fit in the operand stages");
    const size_t smem = sizeof(Smem<BN>) + 1024;
    int rc = smem_limit_once(reinterpret_cast<const void *>(&w4a16_umma_kernel<BN>), (int)smem);
    if (rc) return rc;
    const int n_tiles = (N + kTileN - 1) / kTileN, token_tiles = (M + BN - 1) / BN, G = K / kGroup;
    // split the groups over a cluster (2, 4 or 8 CTAs: sizes that pack into
    // the GPCs) when the tiles alone leave SMs idle
    int C = 1;
    while (C < 8 && n_tiles * token_tiles * C * 2 <= sm_count() && 2 * C * 2 <= G) C *= 2;
    dim3 grid((unsigned)(n_tiles * C), (unsigned)token_tiles);
    if (C == 1)
        return launch_pdl("qspec_linear_w4a16", w4a16_umma_kernel<BN>, grid, dim3(kThreads), smem, stream, x, ldx,
                          packed, sz, M, N, K, y, ldy, st, C, wait_limit, stall, kv);
    return launch_pdl_cluster("qspec_linear_w4a16", w4a16_umma_kernel<BN>, grid, dim3(kThreads), smem, stream, C, x,
                              ldx, packed, sz, M, N, K, y, ldy, st, C, wait_limit, stall, kv);
}

}  // namespace

// Large-M W4A16: token tile 32, 64, 96 or 128 (larger M: several token tiles).
int launch_w4a16_tc(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                    uint16_t *y, int ldy, int32_t *st, cudaStream_t stream, uint32_t wait_limit, int stall,
                    const KvOut &kv) {
    if (M <= 32) return launch_bn<32>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
    if (M <= 64) return launch_bn<64>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
    if (M <= 96) return launch_bn<96>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
    return launch_bn<128>(x, ldx, packed, sz, M, N, K, y, ldy, st, stream, wait_limit, stall, kv);
}

}  // namespace qspec
