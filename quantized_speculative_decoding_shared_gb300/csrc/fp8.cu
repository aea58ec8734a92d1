// fp8.cu -- the SpecQuant Q8 variant: FP8 (E4M3) weights derived from the
// FP16 parent, per-token E4M3 activations, and the FP8 linear of the Q8
// (parent / verify) model on the Blackwell tensor cores.
//
// SpecQuant summary page ("SpecQuant: Speculative Decoding with Multi-Parent
// Quantization for Adaptive LLM Inference"), contributions and approach: Q4
// (INT4), Q8 (FP8) and Q16 (FP16) are derived post-training from one FP16
// parent with shared base weights; the chosen parent verifies the draft.
// Definitions (the same as the CPU oracle's):
//   s = amax / 448 per row (fp32, IEEE division), code = E4M3(v / s) (fp32
//   IEEE quotient, round to nearest even, saturated at 448; a zero row has
//   s = 0 and codes 0); weights per output channel, activations per token;
//   y[m][n] = bf16((sum_k E4M3(xq) E4M3(w8)) sa[m] s8[n]), the sum in fp32.
//
// The linear: one CTA per 128 output channels x BN tokens; both operands are
// streamed by TMA in 128 x 128-byte boxes with 128-byte swizzle (the K-major
// layout the MMA descriptor reads directly: 8 rows x 128 bytes per 1024-byte
// atom, a K step of 32 bytes advancing the start address), a ring of S
// stages.  Warp 4 (one lane) issues the copies -- the weight boxes of the
// first stages before the dependency wait, the weights being immutable --
// warp 5 (one lane) issues 4 MMAs kind::f8f6f4 (M = 128, N = BN, K = 32) per
// stage into one fp32 accumulator in tensor memory, and warps 0-3 (thread =
// TMEM lane = output channel) scale and store it at the end.  A CTA uses at
// most ~110 KB of shared memory and BN (>= 32) tensor-memory columns, so two
// share an SM and one's start and end overlap the other's streaming.  Every wait is
// bounded (QSPEC_ERR_TIMEOUT on expiry, then a drain and a clean exit).
#include <algorithm>
#include <cuda_fp8.h>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

namespace f8 {

// ---------------------------------------------------------------------------
// row quantiser: one CTA per row, 8 values per thread and step
// ---------------------------------------------------------------------------
constexpr int kQThreads = 256;

__device__ __forceinline__ uint8_t e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// kHalf: fp16 input (the parent weights), else bf16 (activations)
template <bool kHalf>
__global__ void __launch_bounds__(kQThreads)
    quant_rows_kernel(const uint16_t *__restrict__ in, int K, int ld, uint8_t *__restrict__ out,
                      float *__restrict__ scale, int32_t *__restrict__ st) {
    __shared__ float red[kQThreads / 32];
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4 *row = reinterpret_cast<const uint4 *>(in + (size_t)r * ld);
    pdl_launch_dependents();
    pdl_wait();
    auto val = [&](uint32_t bits) {
        return kHalf ? __half2float(__ushort_as_half((uint16_t)bits)) : bf16_bits_to_float(bits);
    };
    float amax = 0.0f;
    bool bad = false;
    for (int i = threadIdx.x; i < K / 8; i += kQThreads) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = val(w[e] & 0xFFFF), b = val(w[e] >> 16);
            bad |= !isfinite(a) || !isfinite(b);
            amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    const int bad_any = __syncthreads_or(bad ? 1 : 0);
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 448.0f);
    for (int i = threadIdx.x; i < K / 8; i += kQThreads) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t c0 = s == 0.0f ? 0u : e4m3(__fdiv_rn(val(w[e] & 0xFFFF), s));
            const uint32_t c1 = s == 0.0f ? 0u : e4m3(__fdiv_rn(val(w[e] >> 16), s));
            const uint32_t pair = c0 | (c1 << 8);
            if (e < 2)
                lo |= pair << (16 * e);
            else
                hi |= pair << (16 * (e - 2));
        }
        reinterpret_cast<uint2 *>(out + (size_t)r * K)[i] = make_uint2(lo, hi);
    }
    if (threadIdx.x == 0) {
        scale[r] = s;
        if (bad_any) flag(st, QSPEC_ERR_NONFINITE);
    }
}

// ---------------------------------------------------------------------------
// the FP8 linear
// ---------------------------------------------------------------------------
constexpr int kTileN = 128;                 // output channels per CTA (MMA M)
constexpr int kKB = 128;                    // K per stage: 128 E4M3 bytes
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr size_t kSmemBudget = 110 * 1024;   // two CTAs per SM: one's start and end overlap the other's stream

// shared-memory descriptor of a K-major operand in the 128-byte swizzled
// layout: start address, leading offset unused (16 bytes), stride 1024 bytes
// between 8-row groups, descriptor version 1, swizzle mode 2 (128 bytes)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

template <int BN>
constexpr int stage_bytes() { return kTileN * kKB + BN * kKB; }

template <int BN>
__global__ void __launch_bounds__(kThreads, 2)
    fp8_umma_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                    const float *__restrict__ sa, const float *__restrict__ s8, int M, int N, int K,
                    uint16_t *__restrict__ y, int ldy, int32_t *__restrict__ st, int S, uint32_t wait_limit) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kStage = stage_bytes<BN>();
    constexpr uint32_t kCols = BN < 32 ? 32 : BN;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * kStage);
    uint64_t *empty = full + S, *done = empty + S;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ int timeout_flag;
    __shared__ uint64_t drain_bar;
    volatile int *timeout = &timeout_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileN, t0 = blockIdx.y * BN;
    const int nk = K / kKB;
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (*timeout) return false;
        if (umma::mbar_wait(bar, parity, wait_limit)) return true;
        *timeout = 1;
        return false;
    };

    if (threadIdx.x == 0) {
        *timeout = 0;
        for (int i = 0; i < S; ++i) {
            umma::mbar_init(&full[i], 1);
            umma::mbar_init(&empty[i], 1);
        }
        umma::mbar_init(done, 1);
        umma::mbar_init(&drain_bar, 1);
        umma::mbar_fence_init();
    }
    if (warp == kMmaWarp) umma::tmem_alloc(tslot, kCols);
    if (warp == kProducerWarp && lane == 0) {
        umma::prefetch_tmap(&tw);
        umma::prefetch_tmap(&tx);
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    pdl_launch_dependents();
    const uint32_t tbase = *tslot;
    int issued_k = 0;                          // K blocks whose MMAs were issued (MMA lane 0)
    int loads = 0;                             // stages whose copies were issued (producer lane 0)

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // the first stages' weight boxes before the dependency wait, then
            // their activation boxes; one barrier per stage counts both
            const int pre = min(S, nk);
            for (int i = 0; i < pre; ++i) {
                uint8_t *stg = smem + (size_t)i * kStage;
                umma::mbar_arrive_expect_tx(&full[i], kStage);
                umma::tma_load_2d(stg, &tw, i * kKB, n0, &full[i]);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i)
                umma::tma_load_2d(smem + (size_t)i * kStage + kTileN * kKB, &tx, i * kKB, t0, &full[i]);
            loads = pre;
            for (int i = pre; i < nk; ++i) {
                const int s = i % S;
                if (!wait(&empty[s], (uint32_t)(((i / S) + 1) & 1))) break;
                uint8_t *stg = smem + (size_t)s * kStage;
                umma::mbar_arrive_expect_tx(&full[s], kStage);
                umma::tma_load_2d(stg, &tw, i * kKB, n0, &full[s]);
                umma::tma_load_2d(stg + kTileN * kKB, &tx, i * kKB, t0, &full[s]);
                loads = i + 1;
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma::instr_desc(0, 0, kTileN, BN);   // e4m3 x e4m3 -> f32
            for (int i = 0; i < nk; ++i) {
                const int s = i % S;
                if (!wait(&full[s], (uint32_t)((i / S) & 1))) break;
                umma::fence_after_sync();
                const uint32_t a = umma::smem_addr(smem + (size_t)s * kStage);
                const uint64_t ad = desc_sw128(a), bd = desc_sw128(a + kTileN * kKB);
#pragma unroll
                for (int kk = 0; kk < kKB / 32; ++kk)      // K = 32 bytes per MMA: +2 in the address field
                    umma::mma_e4m3(tbase, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0 ? 1u : 0u);
                umma::mma_commit(&empty[s]);
                issued_k = i + 1;
            }
            if (issued_k == nk) umma::mma_commit(done);
        }
    } else {
        // ---- epilogue: thread = TMEM lane = output channel ----
        pdl_wait();
        if (wait(done, 0)) {
            umma::fence_after_sync();
            const int n = n0 + 32 * warp + lane;
            const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
            const float sn = n < N ? s8[n] : 0.0f;
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t d[16];
                umma::tmem_ld_cols<16>(tbase + lane_off + c0, d);
                umma::tmem_ld_wait();
                if (n < N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = t0 + c0 + j;
                        if (m < M)
                            y[(size_t)m * ldy + n] =
                                float_to_bf16_bits(__fmul_rn(__fmul_rn(__uint_as_float(d[j]), sa[m]), sn));
                    }
                }
            }
        }
    }

    // after a timeout: the copies and MMAs in flight finish (bounded) before
    // the shared and tensor memory are released; the producer and the MMA
    // issuer stopped issuing at the timeout, so at most S copies per stage
    // are outstanding
    __syncthreads();
    if (*timeout) {
        if (warp == kProducerWarp && lane == 0)
            for (int b = max(0, loads - S); b < loads; ++b)
                umma::mbar_wait(&full[b % S], (uint32_t)((b / S) & 1), kWaitLimit);
        if (warp == kMmaWarp && lane == 0 && issued_k > 0) {
            umma::mma_commit(&drain_bar);
            umma::mbar_wait(&drain_bar, 0, kWaitLimit);
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *timeout) flag(st, QSPEC_ERR_TIMEOUT);
    if (warp == kMmaWarp) umma::tmem_free(tbase, kCols);
}

template <int BN>
int launch_linear(const uint8_t *xq, const float *sa, const uint8_t *w8, const float *s8, int M, int N, int K,
                  uint16_t *y, int ldy, int32_t *dev_status, cudaStream_t stream) {
    CUtensorMap tw, tx;
    if (byte_tmap_sw128(&tw, w8, N, K, (size_t)K, kTileN) || byte_tmap_sw128(&tx, xq, M, K, (size_t)K, BN))
        return QSPEC_ERR_UNSUPPORTED;
    constexpr int kStage = stage_bytes<BN>();
    const int S = std::min(8, (int)((kSmemBudget - 512) / kStage));
    const size_t smem = (size_t)S * kStage + (size_t)(2 * S + 1) * 8 + 16;
    auto kern = fp8_umma_kernel<BN>;
    int rc = smem_limit_once(reinterpret_cast<const void *>(kern), (int)kSmemBudget);
    if (rc) return rc;
    dim3 grid((unsigned)((N + kTileN - 1) / kTileN), (unsigned)((M + BN - 1) / BN));
    return launch_pdl("qspec_linear_fp8", kern, grid, dim3(kThreads), smem, stream, tw, tx, sa, s8, M, N, K, y, ldy,
                      dev_status, S, kWaitLimit);
}

}  // namespace f8

}  // namespace

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_quant_weights_fp8(const uint16_t *w_fp16, int N, int K, uint8_t *w8, float *s8,
                                       int32_t *dev_status, qspec_stream_t stream) {
    if (!w_fp16 || !w8 || !s8) return QSPEC_ERR_NULL;
    if (N < 1 || K < kGroup || K % kGroup) return QSPEC_ERR_SHAPE;
    if (!aligned(w_fp16, 16) || !aligned(w8, 8) || !aligned(s8, 4)) return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return launch_pdl("qspec_quant_weights_fp8", f8::quant_rows_kernel<true>, dim3((unsigned)N),
                      dim3(f8::kQThreads), 0, as_cuda(stream), w_fp16, K, K, w8, s8, dev_status);
}

extern "C" int qspec_quant_act_fp8(const uint16_t *x_bf16, int M, int K, int ldx, uint8_t *xq, float *sa,
                                   int32_t *dev_status, qspec_stream_t stream) {
    if (!x_bf16 || !xq || !sa) return QSPEC_ERR_NULL;
    if (M < 1 || K < kGroup || K % kGroup || ldx < K) return QSPEC_ERR_SHAPE;
    if (!aligned(x_bf16, 16) || ldx % 8 || !aligned(xq, 8) || !aligned(sa, 4)) return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return launch_pdl("qspec_quant_act_fp8", f8::quant_rows_kernel<false>, dim3((unsigned)M), dim3(f8::kQThreads),
                      0, as_cuda(stream), x_bf16, K, ldx, xq, sa, dev_status);
}

extern "C" int qspec_linear_fp8(const uint8_t *xq, const float *sa, const uint8_t *w8, const float *s8, int M, int N,
                                int K, uint16_t *y_bf16, int ldy, int32_t *dev_status, qspec_stream_t stream) {
    if (!xq || !sa || !w8 || !s8 || !y_bf16) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < kGroup || K % kGroup || ldy < N) return QSPEC_ERR_SHAPE;
    if (!aligned(xq, 16) || !aligned(w8, 16) || !aligned(sa, 4) || !aligned(s8, 4) || !aligned(y_bf16, 2))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    if (M <= 16) return f8::launch_linear<16>(xq, sa, w8, s8, M, N, K, y_bf16, ldy, dev_status, st);
    if (M <= 32) return f8::launch_linear<32>(xq, sa, w8, s8, M, N, K, y_bf16, ldy, dev_status, st);
    if (M <= 64) return f8::launch_linear<64>(xq, sa, w8, s8, M, N, K, y_bf16, ldy, dev_status, st);
    return f8::launch_linear<128>(xq, sa, w8, s8, M, N, K, y_bf16, ldy, dev_status, st);
}
