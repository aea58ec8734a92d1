// w4a16.cu -- a4: W4A16 linear, y = x W^T with W^ = s (W - z), fp32
// accumulation, bf16 output.
//
// QSPEC summary page, background terms: "W4A16" stores weights in 4 bits and
// keeps 16-bit activations, dequantising the weights for the matmul,
// W^ = s (W_INT4 - z); "QSPEC structure": the verify pass over the gamma + 1
// candidate rows of every sequence.
//
// Small-M path (decode verify, M <= 16): warp MMA m16n8k16 bf16 with fp32
// accumulation; the weight tile is the MMA's A operand (16 output channels x
// 16 k), the tokens its B operand (16 k x 8 tokens).  Dequantisation is split
// so the tensor core sees exact small integers:
//   - a code c becomes the bf16 value 128 + c by OR-ing it into the mantissa
//     of 128.0 (bits 0x4300 | c); no conversion instruction is needed;
//   - per group g the accumulator starts at -128 X_g (X_g = sum of the
//     group's activations), so the MMAs leave D = sum_k c_k x_k, and the
//     epilogue adds s_g (D - z_g X_g), which is sum_k s_g (c_k - z_g) x_k.
// The k order inside the MMA is one permutation applied to both operands:
// the tokens' bf16 pairs are permuted once per CTA into shared memory, and
// each thread's 16-byte weight loads feed its A fragments directly.
//
// Work split as in the small-M W4A4 kernel: persistent CTAs over 16-row
// tiles; an item is a tile and a pair of adjacent groups; the 8 warps split a
// tile's pairs and keep fp32 partial sums in registers; at the end of a tile
// the partials go to shared memory (double-buffered) and one warp adds the 8
// warps' partials in a fixed order and stores bf16.  Larger M: tcgen05
// (w4a16_tc.cu).
#include <algorithm>
#include <type_traits>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

namespace {


__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one weight word (codes c0..c7 in nibbles 0..7) -> bf16 pairs of 128 + c:
// (c0, c4), (c1, c5), (c2, c6), (c3, c7)
__device__ __forceinline__ void codes_bf16(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
    p[0] = (w & mask) | magic;
    p[1] = ((w >> 4) & mask) | magic;
    p[2] = ((w >> 8) & mask) | magic;
    p[3] = ((w >> 12) & mask) | magic;
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

// shared memory: token fragments uint4 [slots][G * 16 + 4] (bf16 pairs, k
// permuted, padded so two tokens of a lane phase hit different banks; slots =
// min(MT, M), the most tokens a CTA holds), 16 zero uint4 for the lanes of
// absent tokens, X float [G][MT], partial sums float [2][warps][16][MT]
inline size_t smem_bytes(int MT, int M, int K, int warps) {
    const size_t G = (size_t)K / kGroup, slots = (size_t)std::min(MT, M);
    return slots * (G * 16 + 4) * 16 + 16 * 16 + (size_t)G * MT * 4 + (size_t)2 * warps * 16 * MT * 4;
}

// One item: a 16-row tile and a pair of adjacent groups (g0, g0 + 1), the
// thread's 16-byte pieces of rows r, r + 8 and their scale words.
struct Item {
    uint4 w00, w01, w10, w11;     // [row r / r + 8][group g0 / g0 + 1]
    uint32_t z00, z01, z10, z11;
};

// kWarps: 8 (two CTAs per SM) or 16 (one CTA per SM when the token
// fragments are large)
template <int MT, int kPrefetch, int kWarps>
__global__ void __launch_bounds__(kWarps * 32, 16 / kWarps)
    w4a16_hmma_gemv_kernel(const uint16_t *__restrict__ x, int ldx, const uint8_t *__restrict__ packed,
                           const uint32_t *__restrict__ sz, int M, int N, int K, uint16_t *__restrict__ y,
                           int ldy, KvOut kv) {
    static_assert(MT >= 1 && MT <= 8 && (MT == 1 || MT % 2 == 0), "one n8 block of tokens");
    constexpr int kThreads = kWarps * 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = K / kGroup;
    const int P = (G + 1) / 2;
    const size_t tstride = (size_t)G * 16 + 4;
    uint4 *bfr = reinterpret_cast<uint4 *>(smem_raw);
    uint4 *zero = bfr + (size_t)min(MT, M) * tstride;
    float *xg = reinterpret_cast<float *>(zero + 16);
    float *red = xg + (size_t)G * MT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qr = lane >> 2, qc = lane & 3;
    const int tok0 = blockIdx.y * MT;
    const int n_tiles = (N + 15) / 16;
    const size_t row_bytes = (size_t)K / 2;
    const int ngw = warp < P ? (P - warp + kWarps - 1) / kWarps : 0;   // this warp's pairs per tile
    const int my_tiles = (int)blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int n_items = ngw * my_tiles;
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
    auto load_item = [&](const Prod &c, Item &it) {
        const int g0 = 2 * (warp + c.j * kWarps);
        const int d1 = g0 + 1 < G ? 1 : 0;                       // an odd last group pairs with itself
        const uint4 *a = reinterpret_cast<const uint4 *>(c.p0 + (size_t)g0 * 64);
        const uint4 *b = reinterpret_cast<const uint4 *>(c.p1 + (size_t)g0 * 64);
        it.w00 = ldg_stream(a);
        it.w01 = ldg_stream(a + d1 * 4);
        it.w10 = ldg_stream(b);
        it.w11 = ldg_stream(b + d1 * 4);
        if (z64) {
            const uint2 za = __ldg(reinterpret_cast<const uint2 *>(c.z0 + g0));
            const uint2 zb = __ldg(reinterpret_cast<const uint2 *>(c.z1 + g0));
            it.z00 = za.x;
            it.z01 = za.y;
            it.z10 = zb.x;
            it.z11 = zb.y;
        } else {
            it.z00 = __ldg(c.z0 + g0);
            it.z01 = __ldg(c.z0 + g0 + d1);
            it.z10 = __ldg(c.z1 + g0);
            it.z11 = __ldg(c.z1 + g0 + d1);
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

    // token fragments, one thread per 8 activations; the 16 words of a group
    // sit in 16 consecutive lanes, which reduce the group sum X_g
    const int mt_real = min(MT, M - tok0);
    const int wpr = K / 8;
    constexpr int kBatch = 4;                              // loads in flight per thread
    for (int base = 0; base < mt_real * wpr; base += kBatch * kThreads) {
        uint4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = base + b * kThreads + threadIdx.x;
            const int t = i / wpr, wi = i - t * wpr;
            v[b] = i < mt_real * wpr ? *reinterpret_cast<const uint4 *>(x + (size_t)(tok0 + t) * ldx + (size_t)wi * 8)
                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = base + b * kThreads + threadIdx.x;
            const bool valid = i < mt_real * wpr;
            const int t = valid ? i / wpr : 0, wi = i - t * wpr;
            const uint4 w = v[b];
            float part = ((bf16_bits_to_float(w.x & 0xFFFF) + bf16_bits_to_float(w.x >> 16)) +
                          (bf16_bits_to_float(w.y & 0xFFFF) + bf16_bits_to_float(w.y >> 16))) +
                         ((bf16_bits_to_float(w.z & 0xFFFF) + bf16_bits_to_float(w.z >> 16)) +
                          (bf16_bits_to_float(w.w & 0xFFFF) + bf16_bits_to_float(w.w >> 16)));
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (valid) {
                const int g = wi >> 4, qcw = (wi >> 2) & 3, u = wi & 3;
                bfr[(size_t)t * tstride + (g * 4 + u) * 4 + qcw] =
                    make_uint4(__byte_perm(w.x, w.z, 0x5410), __byte_perm(w.x, w.z, 0x7632),
                               __byte_perm(w.y, w.w, 0x5410), __byte_perm(w.y, w.w, 0x7632));
                if ((wi & 15) == 0) xg[g * MT + t] = part;
            }
        }
    }
    for (int i = threadIdx.x; i < 16; i += kThreads) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < G * MT; i += kThreads)
        if (i % MT >= mt_real) xg[i] = 0.0f;
    __syncthreads();

    // lanes of absent token columns read the zero words for every group
    const bool present = qr < mt_real;
    const uint4 *brow = present ? bfr + (size_t)qr * tstride + qc : zero + qc;
    const int gstride = present ? 16 : 0;
    // this lane's D columns are tokens 2 qc, 2 qc + 1 (clamped for the
    // X loads; columns past MT are never stored)
    const int tq = MT == 1 ? 0 : (2 * qc < MT ? 2 * qc : 0);

    // end of tile `step`: partials are in red[step & 1]; one warp adds them
    auto tile_done = [&](int step) {
        __syncthreads();
        if (warp != (step & (kWarps - 1))) return;
        const int tile = blockIdx.x + step * gridDim.x;
        const float *rb = red + (size_t)(step & 1) * kWarps * 16 * MT;
        for (int p = lane; p < 16 * MT; p += 32) {
            const int r = p / MT, t = p - (p / MT) * MT, n = tile * 16 + r, m = tok0 + t;
            if (n >= N || m >= M) continue;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += rb[(size_t)w * 16 * MT + p];
            const uint16_t v16 = float_to_bf16_bits(sum);
            y[(size_t)m * ldy + n] = v16;
            kv_store(kv, m, n, v16);
        }
    };
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    auto flush = [&](int step) {                          // this warp's partials of tile `step`
        float *rw = red + (size_t)(step & 1) * kWarps * 16 * MT + (size_t)warp * 16 * MT;
        if (2 * qc < MT) {
            rw[qr * MT + 2 * qc] = acc[0];
            rw[(qr + 8) * MT + 2 * qc] = acc[2];
            if (MT > 1) {
                rw[qr * MT + 2 * qc + 1] = acc[1];
                rw[(qr + 8) * MT + 2 * qc + 1] = acc[3];
            }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
    };

    // group g: D starts at -128 X_g, so after the MMAs D = sum c x
    auto group = [&](const uint4 &wr0, const uint4 &wr1, uint32_t za, uint32_t zb, int g) {
        float X0, X1;
        if (MT == 1) {
            X0 = X1 = xg[g];
        } else {
            const float2 o = *reinterpret_cast<const float2 *>(xg + g * MT + tq);
            X0 = o.x;
            X1 = o.y;
        }
        float d[4] = {-128.0f * X0, -128.0f * X1, -128.0f * X0, -128.0f * X1};
        const uint4 *bf = brow + (size_t)g * gstride;
        const uint32_t w0[4] = {wr0.x, wr0.y, wr0.z, wr0.w}, w1[4] = {wr1.x, wr1.y, wr1.z, wr1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 b = bf[u * 4];
            uint32_t a0[4], a1[4];
            codes_bf16(w0[u], a0);
            codes_bf16(w1[u], a1);
            mma_bf16_16816(d, a0[0], a1[0], a0[1], a1[1], b.x, b.y);
            mma_bf16_16816(d, a0[2], a1[2], a0[3], a1[3], b.z, b.w);
        }
        const float sa = half_lo(za), zfa = half_hi(za), sb = half_lo(zb), zfb = half_hi(zb);
        acc[0] = __fmaf_rn(sa, __fmaf_rn(-zfa, X0, d[0]), acc[0]);
        acc[2] = __fmaf_rn(sb, __fmaf_rn(-zfb, X0, d[2]), acc[2]);
        if (MT > 1) {
            acc[1] = __fmaf_rn(sa, __fmaf_rn(-zfa, X1, d[1]), acc[1]);
            acc[3] = __fmaf_rn(sb, __fmaf_rn(-zfb, X1, d[3]), acc[3]);
        }
    };

    // with an even group count the second group of an item needs no test, so
    // the two groups' unpack and MMAs form one straight block
    auto consume = [&](auto even_tag) {
        constexpr bool evenG = decltype(even_tag)::value;      // every item holds two groups
        int cj = 0, cstep = 0;                                 // consumer cursor
        int cur = 0;                                           // tile step being produced
        for (int base = 0; base < n_items; base += kPrefetch) {
#pragma unroll
            for (int p = 0; p < kPrefetch; ++p) {
                const int it = base + p;
                if (it >= n_items) break;
                if (cstep != cur) {                            // this warp's first item of the next tile
                    flush(cur);
                    tile_done(cur);
                    cur = cstep;
                }
                const int g0 = 2 * (warp + cj * kWarps);
                const Item c = ring[p];
                if (it + kPrefetch < n_items) {
                    load_item(pc, ring[p]);
                    advance_prod(pc);
                }
                group(c.w00, c.w10, c.z00, c.z10, g0);
                if (evenG || g0 + 1 < G) group(c.w01, c.w11, c.z01, c.z11, g0 + 1);
                if (++cj == ngw) {
                    cj = 0;
                    ++cstep;
                }
            }
        }
        return cur;
    };
    int cur = (G % 2 == 0) ? consume(std::true_type()) : consume(std::false_type());
    // the last tile with items, then the remaining ones (warps without pairs)
    for (; cur < my_tiles; ++cur) {
        flush(cur);
        tile_done(cur);
    }
}

template <int MT, int kWarps>
int launch_w4a16_w(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                   uint16_t *y, int ldy, const KvOut &kv, cudaStream_t st) {
    const size_t smem = smem_bytes(MT, M, K, kWarps);
    auto kern = w4a16_hmma_gemv_kernel<MT, 1, kWarps>;
    int rc = smem_limit_once(reinterpret_cast<const void *>(kern), 200 * 1024);
    if (rc) return rc;
    const int n_tiles = (N + 15) / 16, token_tiles = (M + MT - 1) / MT;
    const int per_col = std::max(1, (16 / kWarps) * sm_count() / token_tiles);
    dim3 grid((unsigned)std::min(n_tiles, per_col), (unsigned)token_tiles);
    return launch_pdl("qspec_linear_w4a16", kern, grid, dim3(kWarps * 32), smem, st, x, ldx, packed, sz, M, N, K, y,
                      ldy, kv);
}

// two 8-warp CTAs per SM when their shared memory fits, else one of 16 warps
template <int MT>
int launch_w4a16(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                 uint16_t *y, int ldy, const KvOut &kv, cudaStream_t st) {
    if (smem_bytes(MT, M, K, 8) <= 112 * 1024)
        return launch_w4a16_w<MT, 8>(x, ldx, packed, sz, M, N, K, y, ldy, kv, st);
    return launch_w4a16_w<MT, 16>(x, ldx, packed, sz, M, N, K, y, ldy, kv, st);
}

}  // namespace

}  // namespace qspec

using namespace qspec;

// the W4A16 linear, with the cache output of `kv` when it names a cache
static int linear_w4a16(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N,
                        int K, uint16_t *y_bf16, int ldy, const KvOut &kv, int32_t *dev_status, cudaStream_t st) {
    if (M <= 16) {
        // tokens per CTA: up to 8 (one MMA column block), halved while the
        // token fragments do not fit
        int mt = M == 1 ? 1 : M == 2 ? 2 : M <= 4 ? 4 : 8;
        while (mt > 1 && smem_bytes(mt, M, K, 16) > 200 * 1024) mt /= 2;
        if (smem_bytes(mt, M, K, 16) <= 200 * 1024) {
            switch (mt) {
                case 1: return launch_w4a16<1>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, kv, st);
                case 2: return launch_w4a16<2>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, kv, st);
                case 4: return launch_w4a16<4>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, kv, st);
                default: return launch_w4a16<8>(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, kv, st);
            }
        }
    }
    return launch_w4a16_tc(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, dev_status, st, kWaitLimit, 0, kv);
}

static int w4a16_args(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N,
                      int K, const uint16_t *y_bf16, int ldy) {
    if (!x_bf16 || !packed || !sz || !y_bf16) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < kGroup || K % kGroup || ldx < K || ldy < N) return QSPEC_ERR_SHAPE;
    if (!aligned(x_bf16, 16) || ldx % 8 || !aligned(packed, 16) || !aligned(sz, 4) || !aligned(y_bf16, 2))
        return QSPEC_ERR_ALIGN;
    return check_device();
}

extern "C" int qspec_linear_w4a16(const uint16_t *x_bf16, int ldx, const uint8_t *packed,
                                  const uint32_t *sz, int M, int N, int K, uint16_t *y_bf16,
                                  int ldy, int32_t *dev_status, qspec_stream_t stream) {
    int rc = w4a16_args(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy);
    if (rc) return rc;
    const KvOut none = {nullptr, nullptr, nullptr, nullptr, 0, 1, 1, 1, 0, nullptr};
    return linear_w4a16(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, none, dev_status, as_cuda(stream));
}

extern "C" int qspec_linear_w4a16_kv(const uint16_t *x_bf16, int ldx, const uint8_t *packed, const uint32_t *sz,
                                     int M, int N, int K, uint16_t *y_bf16, int ldy, int kv_col0, int H, int D, int T,
                                     int gamma, uint16_t *k_cache, uint16_t *v_cache, const int32_t *base_pos,
                                     const int32_t *n_acc, int32_t *dev_status, qspec_stream_t stream) {
    int rc = w4a16_args(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy);
    if (rc) return rc;
    if ((!k_cache && !v_cache) || !base_pos) return QSPEC_ERR_NULL;
    if (gamma < 1 || gamma > QSPEC_MAX_GAMMA || M % (gamma + 1) || H < 1 || D < 1 || T < 1 || kv_col0 < 0 ||
        kv_col0 + (v_cache ? 2 : 1) * H * D > N)
        return QSPEC_ERR_SHAPE;
    if ((k_cache && !aligned(k_cache, 2)) || (v_cache && !aligned(v_cache, 2)) || !aligned(base_pos, 4) ||
        (n_acc && !aligned(n_acc, 4)))
        return QSPEC_ERR_ALIGN;
    const KvOut kv = {k_cache, v_cache, base_pos, n_acc, kv_col0, H, D, T, gamma, dev_status};
    return linear_w4a16(x_bf16, ldx, packed, sz, M, N, K, y_bf16, ldy, kv, dev_status, as_cuda(stream));
}
