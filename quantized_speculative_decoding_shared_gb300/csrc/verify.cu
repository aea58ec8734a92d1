// verify.cu -- a5 greedy and a6 sampled verification of gamma draft tokens,
// and draft-side sampling with the draft statistics.
//
// QSPEC summary page, background terms: speculative sampling accepts a draft
// x with probability min(1, p(x|h) / q(x|h)); greedy decoding accepts it when
// it is the target's top-1 token; nothing after the first rejection is kept;
// the target then supplies one more token (a correction drawn from the
// normalised residual max(0, p - q), or a bonus token from the last target
// row when every draft is accepted), so L = A + 1 tokens are emitted.
// "QSPEC structure": the verify pass yields gamma + 1 target distributions.
//
// All decisions are integer so they are reproducible bit for bit:
//   E_v = rint(qexp(l_v - row max) * 2^32), S = sum_v E_v (exact in uint64);
//   accept draft i iff U_i * Eq_t * Sp < 2^24 * Ep_t * Sq (128-bit);
//   residual R_v = max(0, Ep_v Sq - Eq_v Sp) (128-bit; the target row's E if
//   every R_v is 0); draw v* = min{v : sum_{u<=v} w_u > floor(U' sum w / 2^24)}.
// Integer sums are associative, so rows are split into chunks processed by
// many CTAs and combined with atomics without changing a single bit.
//
// Launch sequence (one stream, no host synchronisation):
//   greedy : argmax (chunk x row, one chunk per row when there are at
//            least two rows per SM; one key per chunk), finalize (per
//            sequence: max over the chunk keys, first mismatch)
//   sampled: row max and row sums (one CTA per row, the second pass over the
//            row hitting L2; else memset, then chunk x row kernels for each
//            with atomics), decisions + residual chunk sums (chunk x
//            sequence), draw (per sequence)
//   draft  : rows of at least kDraftClusterMinV logits and fewer than two
//            rows per SM: one launch, a cluster of 16 CTAs per row
//            (each a slice of the row; the slices' maxima, weight sums and
//            entropy parts exchanged through distributed shared memory, the
//            draw in the slice that holds the threshold); otherwise the same
//            row statistics as above over the B draft rows, weight sums and
//            entropy parts (chunk x row), the draw on the row's own weights
//            (Philox slot 16 + step), the features (per row).  SpecKV blog,
//            architecture section: the confidence and entropy of the draft
//            softmax are the features its gamma controller reads.
// HBM traffic: one read of every logit (B (2 gamma + 1) V bf16) plus L2
// re-reads of the rows a later phase needs.
#include <algorithm>
#include <type_traits>

#include <mutex>

#include "qspec_device.cuh"
#include "qspec_host.h"
#include "umma.cuh"

namespace qspec {

namespace {

constexpr int kThreads = 256;
constexpr int kSub = kThreads * 8;    // elements one CTA covers per pass (8 per thread)
constexpr int kMaxChunks = 256;
// greedy: rows x chunks keys, with chunks sized for about two CTAs per SM,
// fit in rows + kGreedyExtraKeys slots (for up to 512 SMs)
constexpr int kGreedyExtraKeys = 1024;

struct Layout {
    int chunk;        // elements per chunk (multiple of kSub)
    int n_chunks;     // <= kMaxChunks
    size_t off_key, off_max, off_sum, off_rsum, off_esum, off_acc, total;
};

inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

Layout make_layout(int B, int gamma, int V) {
    Layout L;
    int subs = (V + kSub - 1) / kSub;
    int per = (subs + kMaxChunks - 1) / kMaxChunks;
    L.chunk = per * kSub;
    L.n_chunks = (V + L.chunk - 1) / L.chunk;
    size_t rows_g = (size_t)B * (gamma + 1), rows_s = (size_t)B * (2 * gamma + 1);
    size_t o = 0;
    L.off_key = o;  o = align16(o + (rows_g + kGreedyExtraKeys) * 8); // greedy (row, chunk) argmax keys
    L.off_max = o;  o = align16(o + rows_s * 4);                 // row max, ordered bits
    L.off_sum = o;  o = align16(o + rows_s * 8);                 // row sums S
    L.off_rsum = o; o = align16(o + (size_t)B * L.n_chunks * 16); // residual chunk sums
    L.off_esum = o; o = align16(o + (size_t)B * L.n_chunks * 8);  // target-row chunk sums
    L.off_acc = o;  o = align16(o + (size_t)B * 4);              // A_b
    L.total = o;
    return L;
}

// -------------------------------------------------------------------------
// Two fixed-point weights at once: the same fp32 operations, rounded the
// same way, as fixed_weight for each element, with the floating-point steps
// as packed f32x2 instructions (each lane rounds exactly as the scalar
// instruction), so the row pass issues fewer instructions per logit.
// -------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ void fixed_weight2(float l0, float l1, float m, uint64_t &w0, uint64_t &w1) {
    const uint64_t x0 = sub2(pk2(l0, l1), pk2(m, m));
    const float xa = lo2(x0) < -32.0f ? -32.0f : lo2(x0), xb = hi2(x0) < -32.0f ? -32.0f : hi2(x0);
    const uint64_t x = pk2(xa, xb);
    const uint64_t magic = pk2(12582912.0f, 12582912.0f);
    const uint64_t t = add2(mul2(x, pk2(__uint_as_float(0x3FB8AA3Bu), __uint_as_float(0x3FB8AA3Bu))), magic);
    const uint64_t nn = sub2(t, magic) ^ 0x8000000080000000ull;           // -n, exactly
    uint64_t r = fma2(nn, pk2(__uint_as_float(0x3F317200u), __uint_as_float(0x3F317200u)), x);
    r = fma2(nn, pk2(__uint_as_float(0x35BFBE8Eu), __uint_as_float(0x35BFBE8Eu)), r);
    uint64_t p = pk2(__uint_as_float(0x39500D01u), __uint_as_float(0x39500D01u));          // 1/7!
    p = fma2(p, r, pk2(__uint_as_float(0x3AB60B61u), __uint_as_float(0x3AB60B61u)));      // 1/6!
    p = fma2(p, r, pk2(__uint_as_float(0x3C088889u), __uint_as_float(0x3C088889u)));      // 1/5!
    p = fma2(p, r, pk2(__uint_as_float(0x3D2AAAABu), __uint_as_float(0x3D2AAAABu)));      // 1/4!
    p = fma2(p, r, pk2(__uint_as_float(0x3E2AAAABu), __uint_as_float(0x3E2AAAABu)));      // 1/3!
    p = fma2(p, r, pk2(0.5f, 0.5f));
    p = fma2(p, r, pk2(1.0f, 1.0f));
    p = fma2(p, r, pk2(1.0f, 1.0f));
    const int ea = (int)(__float_as_uint(lo2(t)) - 0x4B400000u), eb = (int)(__float_as_uint(hi2(t)) - 0x4B400000u);
    const uint64_t v = mul2(p, pk2(__int_as_float((ea + 127 + 32) << 23), __int_as_float((eb + 127 + 32) << 23)));
    const float va = lo2(v), vb = hi2(v);
    const uint64_t wa = va >= 4294967296.0f ? (1ull << 32) : (uint64_t)__float2uint_rn(va);
    const uint64_t wb = vb >= 4294967296.0f ? (1ull << 32) : (uint64_t)__float2uint_rn(vb);
    w0 = lo2(x0) < -32.0f ? 0ull : wa;
    w1 = hi2(x0) < -32.0f ? 0ull : wb;
}

// -------------------------------------------------------------------------
// helpers: load 8 logits of a row starting at element v0 (V % 8 == 0 path,
// else element-wise); missing elements read as -inf.
// -------------------------------------------------------------------------
template <bool VEC>
__device__ __forceinline__ void load8(const uint16_t *row, int v0, int V, float f[8]) {
    if (VEC) {
        if (v0 + 8 <= V) {
            uint4 u = __ldg(reinterpret_cast<const uint4 *>(row + v0));
            uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (v0 + i < V) ? bf16_bits_to_float(row[v0 + i]) : -INFINITY;
}

template <typename T, int NT = kThreads>
__device__ __forceinline__ T block_reduce_max(T v, T *sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        T u = __shfl_xor_sync(0xffffffffu, v, o);
        v = u > v ? u : v;
    }
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < NT / 32 ? sh[threadIdx.x] : sh[0];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            T u = __shfl_xor_sync(0xffffffffu, v, o);
            v = u > v ? u : v;
        }
    }
    __syncthreads();
    return v;   // valid in thread 0
}

template <int NT = kThreads>
__device__ __forceinline__ unsigned long long block_reduce_sum(unsigned long long v,
                                                               unsigned long long *sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < NT / 32 ? sh[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    }
    __syncthreads();
    return v;
}

// inclusive block scan of u128 values (kThreads entries in shared memory)
__device__ __forceinline__ u128 block_scan_u128(u128 v, u128 *buf) {
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < kThreads; off <<= 1) {
        u128 add = threadIdx.x >= off ? buf[threadIdx.x - off] : (u128)0;
        __syncthreads();
        buf[threadIdx.x] += add;
        __syncthreads();
    }
    return buf[threadIdx.x];
}

// -------------------------------------------------------------------------
// greedy
// -------------------------------------------------------------------------
// CTA (row, chunk): the argmax key of P[row][chunk], written to
// keys[row * gridDim.y + chunk]; four 8-logit loads per thread in flight.
// Each thread keeps the first of its largest logits (strict >, increasing
// index, so -0 and +0 tie as in float comparison and NaN never wins),
// starting from its first logit; the key (value with -0 made +0, then the
// lowest index) picks the CTA's winner.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) greedy_argmax_kernel(const uint16_t *__restrict__ P, int V,
                                                                int chunk,
                                                                unsigned long long *__restrict__ keys,
                                                                int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ unsigned long long sh[kThreads / 32];
    const int row = blockIdx.x;
    const uint16_t *rp = P + (size_t)row * V;
    const int c0 = blockIdx.y * chunk, c1 = min(V, c0 + chunk);
    float bv = -INFINITY;
    int bi = c0 + threadIdx.x * 8;                          // its first logit (or none)
    bool bad = false;
    for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += kSub * 4) {
        float f[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) load8<VEC>(rp, v0 + u * kSub, c1, f[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                bad |= isnan(f[u][i]);                    // (missing logits read as -inf)
                if (f[u][i] > bv) {
                    bv = f[u][i];
                    bi = v0 + u * kSub + i;
                }
            }
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
    unsigned long long best = 0;
    if (bi < c1)
        best = ((unsigned long long)ordered_bits(__fadd_rn(bv, 0.0f)) << 32) | (0xFFFFFFFFu - (uint32_t)bi);
    best = block_reduce_max(best, sh);
    if (threadIdx.x == 0) keys[(size_t)row * gridDim.y + blockIdx.y] = best;
}

// per sequence: the row argmaxes (max over the row's nch chunk keys), the
// first mismatch, the emitted tokens
__global__ void greedy_finalize_kernel(const unsigned long long *__restrict__ keys, int nch,
                                       const int32_t *__restrict__ draft, int B, int gamma, int V,
                                       int32_t *__restrict__ n_acc, int32_t *__restrict__ out,
                                       int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    auto row_arg = [&](int i) {
        const unsigned long long *k = keys + ((size_t)b * (gamma + 1) + i) * nch;
        unsigned long long best = 0;
        for (int c = 0; c < nch; ++c) best = k[c] > best ? k[c] : best;
        return (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    };
    const int32_t *d = draft + (size_t)b * gamma;
    int A = gamma;
    bool bad = false;
    for (int i = 0; i < gamma; ++i) {
        int t = d[i];
        bad |= (t < 0 || t >= V);
        if (A == gamma && t != row_arg(i)) A = i;
    }
    if (bad) flag(st, QSPEC_ERR_RANGE);
    int32_t *o = out + (size_t)b * (gamma + 1);
    for (int i = 0; i <= gamma; ++i) o[i] = i < A ? d[i] : -1;
    o[A] = row_arg(A);
    n_acc[b] = A;
}

// -------------------------------------------------------------------------
// sampled: rows 0 .. B(gamma+1)-1 are P[b][i], then B gamma rows of Q[b][i]
// -------------------------------------------------------------------------
__device__ __forceinline__ const uint16_t *row_ptr(const uint16_t *P, const uint16_t *Q, int B,
                                                   int gamma, int V, int row) {
    int np = B * (gamma + 1);
    return row < np ? P + (size_t)row * V : Q + (size_t)(row - np) * V;
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads) sample_rowmax_kernel(const uint16_t *__restrict__ P,
                                                                const uint16_t *__restrict__ Q, int B,
                                                                int gamma, int V, int chunk,
                                                                uint32_t *__restrict__ maxenc,
                                                                int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ uint32_t sh[kThreads / 32];
    const int row = blockIdx.x;
    const uint16_t *rp = row_ptr(P, Q, B, gamma, V, row);
    const int c0 = blockIdx.y * chunk, c1 = min(V, c0 + chunk);
    float m = -INFINITY;
    bool bad = false;
    for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += kSub) {
        float f[8];
        load8<VEC>(rp, v0, c1, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bad |= isnan(f[i]) || f[i] == INFINITY;
            m = fmaxf(m, f[i]);
        }
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
    uint32_t e = block_reduce_max(ordered_bits(m), sh);
    if (threadIdx.x == 0) atomicMax(maxenc + row, e);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads) sample_rowsum_kernel(const uint16_t *__restrict__ P,
                                                                const uint16_t *__restrict__ Q, int B,
                                                                int gamma, int V, int chunk,
                                                                const uint32_t *__restrict__ maxenc,
                                                                unsigned long long *__restrict__ sums,
                                                                int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ unsigned long long sh[kThreads / 32];
    const int row = blockIdx.x;
    const uint16_t *rp = row_ptr(P, Q, B, gamma, V, row);
    const float m = from_ordered_bits(maxenc[row]);
    if (m == -INFINITY) {                      // a row without any mass
        if (blockIdx.y == 0 && threadIdx.x == 0) flag(st, QSPEC_ERR_NONFINITE);
        return;
    }
    const int c0 = blockIdx.y * chunk, c1 = min(V, c0 + chunk);
    unsigned long long s = 0;
    for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += kSub) {
        float f[8];
        load8<VEC>(rp, v0, c1, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += fixed_weight(f[i], m);
    }
    s = block_reduce_sum(s, sh);
    if (threadIdx.x == 0 && s) atomicAdd(sums + row, s);
}

// one CTA of kRowThreads per row (used when there are enough rows to fill the
// GPU): the row maximum, then the sum of fixed weights over the same row.  Two
// CTAs per SM keep 2 x 152 rows in flight, few enough that the second pass
// finds the row in L2.  Both results are written directly (no atomics, no
// cleared workspace); the first pass keeps kUnroll loads in flight per thread.
constexpr int kRowThreads = 512;
constexpr int kUnroll = 4;

// block reduction over kRowThreads threads with operator op and its identity
template <typename T, typename Op>
__device__ __forceinline__ T row_reduce(T v, T *sh, T identity, Op op) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < kRowThreads / 32 ? sh[threadIdx.x] : identity;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    }
    __syncthreads();
    return v;   // valid in thread 0
}

template <bool VEC>
__global__ void __launch_bounds__(kRowThreads, 2) sample_rowstats_kernel(const uint16_t *__restrict__ P,
                                                                        const uint16_t *__restrict__ Q, int B,
                                                                        int gamma, int V,
                                                                        uint32_t *__restrict__ maxenc,
                                                                        unsigned long long *__restrict__ sums,
                                                                        int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kStep = kRowThreads * 8;
    __shared__ uint32_t shm[kRowThreads / 32];
    __shared__ unsigned long long shs[kRowThreads / 32];
    __shared__ uint32_t s_m;
    const int row = blockIdx.x;
    const uint16_t *rp = row_ptr(P, Q, B, gamma, V, row);
    float m = -INFINITY;
    bool bad = false;
    for (int v0 = threadIdx.x * 8; v0 < V; v0 += kStep * kUnroll) {
        float f[kUnroll][8];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) load8<VEC>(rp, v0 + u * kStep, V, f[u]);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                bad |= isnan(f[u][i]) || f[u][i] == INFINITY;
                m = fmaxf(m, f[u][i]);
            }
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
    const uint32_t e =
        row_reduce(ordered_bits(m), shm, 0u, [](uint32_t a, uint32_t b) { return a > b ? a : b; });
    if (threadIdx.x == 0) {
        s_m = e;
        maxenc[row] = e;
    }
    __syncthreads();
    m = from_ordered_bits(s_m);
    if (m == -INFINITY) {                      // a row without any mass
        if (threadIdx.x == 0) {
            flag(st, QSPEC_ERR_NONFINITE);
            sums[row] = 0;
        }
        return;
    }
    unsigned long long sum = 0;
    for (int v0 = threadIdx.x * 8; v0 < V; v0 += kStep * 2) {
        float f[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) load8<VEC>(rp, v0 + u * kStep, V, f[u]);
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                uint64_t w0, w1;
                fixed_weight2(f[u][i], f[u][i + 1], m, w0, w1);
                sum += w0 + w1;
            }
    }
    sum = row_reduce(sum, shs, 0ull, [](unsigned long long a, unsigned long long b) { return a + b; });
    if (threadIdx.x == 0) sums[row] = sum;
}

// decisions of sequence b: A_b (first rejected draft index, gamma if none)
__device__ int decide(const uint16_t *P, const uint16_t *Q, const int32_t *draft, int B, int gamma,
                      int V, int b, uint64_t seed, uint64_t round, const uint32_t *maxenc,
                      const unsigned long long *sums, bool *range_bad) {
    // thread i < gamma tests draft i; result combined with a ballot in warp 0
    int reject = 0;
    bool bad = false;
    if (threadIdx.x < 32) {
        int i = threadIdx.x;
        if (i < gamma) {
            int t = draft[(size_t)b * gamma + i];
            bad = t < 0 || t >= V;
            t = bad ? 0 : t;
            int rp = b * (gamma + 1) + i;
            int rq = B * (gamma + 1) + b * gamma + i;
            float mp = from_ordered_bits(maxenc[rp]), mq = from_ordered_bits(maxenc[rq]);
            uint64_t Ep = fixed_weight(bf16_bits_to_float(P[(size_t)rp * V + t]), mp);
            uint64_t Eq = fixed_weight(bf16_bits_to_float(Q[((size_t)b * gamma + i) * V + t]), mq);
            uint64_t Sp = sums[rp], Sq = sums[rq];
            uint32_t U = uniform24(seed, round, (uint32_t)i, (uint32_t)b);
            u128 lhs = (u128)U * Sp * Eq;
            u128 rhs = ((u128)Ep * Sq) << 24;
            reject = !(lhs < rhs);
        }
        unsigned rj = __ballot_sync(0xffffffffu, reject);
        unsigned bd = __ballot_sync(0xffffffffu, bad);
        *range_bad = bd != 0;
        return rj ? __ffs(rj) - 1 : gamma;
    }
    return -1;
}

// grid (b, chunk): decisions (recomputed by every chunk's CTA), then this
// chunk's sums of the residual R_v and of the target row's E_v.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) sample_residual_kernel(
    const uint16_t *__restrict__ P, const uint16_t *__restrict__ Q, const int32_t *__restrict__ draft,
    int B, int gamma, int V, int chunk, uint64_t seed, uint64_t round,
    const uint32_t *__restrict__ maxenc, const unsigned long long *__restrict__ sums,
    u128 *__restrict__ rsum, unsigned long long *__restrict__ esum, int32_t *__restrict__ accbuf,
    int32_t *__restrict__ n_acc, int32_t *__restrict__ out, int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int sA;
    __shared__ u128 shr[kThreads / 32];
    __shared__ unsigned long long she[kThreads / 32];
    const int b = blockIdx.x;
    const int n_chunks = gridDim.y;
    bool range_bad = false;
    int A = decide(P, Q, draft, B, gamma, V, b, seed, round, maxenc, sums, &range_bad);
    if (threadIdx.x == 0) {
        sA = A;
        if (blockIdx.y == 0) {
            if (range_bad) flag(st, QSPEC_ERR_RANGE);
            accbuf[b] = A;
            n_acc[b] = A;
            int32_t *o = out + (size_t)b * (gamma + 1);
            for (int i = 0; i <= gamma; ++i) o[i] = i < A ? draft[(size_t)b * gamma + i] : -1;
        }
    }
    __syncthreads();
    A = sA;
    const int rp = b * (gamma + 1) + A;
    const float mp = from_ordered_bits(maxenc[rp]);
    const uint64_t Sp = sums[rp];
    const bool residual = A < gamma;
    const int rq = B * (gamma + 1) + b * gamma + (residual ? A : 0);
    const float mq = from_ordered_bits(maxenc[rq]);
    const uint64_t Sq = sums[rq];
    const uint16_t *prow = P + (size_t)rp * V;
    const uint16_t *qrow = Q + ((size_t)b * gamma + (residual ? A : 0)) * V;
    const int c0 = blockIdx.y * chunk, c1 = min(V, c0 + chunk);
    u128 r = 0;
    unsigned long long e = 0;
    // the residual test is uniform over the CTA: one loop for each case, no
    // branch between the elements' weights
    auto walk = [&](auto residual_tag) {
        constexpr bool kRes = decltype(residual_tag)::value;
        for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += kSub) {
            float fp[8], fq[8];
            load8<VEC>(prow, v0, c1, fp);
            if constexpr (kRes) load8<VEC>(qrow, v0, c1, fq);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                uint64_t Ep[2], Eq[2];
                fixed_weight2(fp[i], fp[i + 1], mp, Ep[0], Ep[1]);
                e += Ep[0] + Ep[1];
                if constexpr (kRes) {
                    fixed_weight2(fq[i], fq[i + 1], mq, Eq[0], Eq[1]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        u128 a = (u128)Ep[h] * Sq, c = (u128)Eq[h] * Sp;
                        r += a > c ? a - c : (u128)0;
                    }
                }
            }
        }
    };
    if (residual)
        walk(std::true_type());
    else
        walk(std::false_type());
    // block sums (u128 via two halves with carry handled by the scan helper)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        uint64_t lo = (uint64_t)r, hi = (uint64_t)(r >> 64);
        uint64_t lo2 = __shfl_xor_sync(0xffffffffu, lo, o), hi2 = __shfl_xor_sync(0xffffffffu, hi, o);
        r += ((u128)hi2 << 64) | lo2;
        e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if ((threadIdx.x & 31) == 0) {
        shr[threadIdx.x >> 5] = r;
        she[threadIdx.x >> 5] = e;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        u128 rt = 0;
        unsigned long long et = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            rt += shr[w];
            et += she[w];
        }
        rsum[(size_t)b * n_chunks + blockIdx.y] = rt;
        esum[(size_t)b * n_chunks + blockIdx.y] = et;
    }
}

// one CTA per sequence: pick the chunk holding the draw, then the element.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) sample_draw_kernel(
    const uint16_t *__restrict__ P, const uint16_t *__restrict__ Q, int B, int gamma, int V,
    int chunk, int n_chunks, uint64_t seed, uint64_t round, uint32_t slot, const uint32_t *__restrict__ maxenc,
    const unsigned long long *__restrict__ sums, const u128 *__restrict__ rsum,
    const unsigned long long *__restrict__ esum, const int32_t *__restrict__ accbuf,
    int32_t *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ u128 buf[kThreads];
    __shared__ int s_chunk, s_mode;
    __shared__ u128 s_base;
    const int b = blockIdx.x;
    const int A = accbuf[b];
    const bool residual0 = A < gamma;
    // chunk totals of the residual; fall back to the target row if all zero
    u128 rv = (threadIdx.x < n_chunks && residual0) ? rsum[(size_t)b * n_chunks + threadIdx.x] : (u128)0;
    u128 rinc = block_scan_u128(rv, buf);
    u128 Wr = buf[kThreads - 1];
    __syncthreads();
    const bool residual = residual0 && Wr != 0;
    u128 inc = rinc;
    u128 W = Wr;
    if (!residual) {
        u128 ev = threadIdx.x < n_chunks ? (u128)esum[(size_t)b * n_chunks + threadIdx.x] : (u128)0;
        inc = block_scan_u128(ev, buf);
        W = buf[kThreads - 1];
        __syncthreads();
    }
    const uint32_t U = uniform24(seed, round, slot, (uint32_t)b);
    const u128 T = ((u128)U * W) >> 24;
    // the first chunk whose inclusive prefix exceeds T
    if (threadIdx.x == 0) s_chunk = n_chunks - 1;
    __syncthreads();
    {
        u128 exc = inc - (threadIdx.x < n_chunks ? (residual ? rv
                                                             : (u128)esum[(size_t)b * n_chunks + threadIdx.x])
                                                 : (u128)0);
        if (threadIdx.x < n_chunks && inc > T && exc <= T) {
            s_chunk = threadIdx.x;
            s_base = exc;
        }
    }
    __syncthreads();
    const int c = s_chunk;
    const u128 base = c == 0 ? (u128)0 : s_base;
    // walk chunk c: per-thread sums of 8 consecutive elements, scan, find
    const int rp = b * (gamma + 1) + A;
    const float mp = from_ordered_bits(maxenc[rp]);
    const uint64_t Sp = sums[rp];
    const int rq = B * (gamma + 1) + b * gamma + (residual ? A : 0);
    const float mq = residual ? from_ordered_bits(maxenc[rq]) : 0.0f;
    const uint64_t Sq = residual ? sums[rq] : 0;
    const uint16_t *prow = P + (size_t)rp * V;
    const uint16_t *qrow = Q + ((size_t)b * gamma + (residual ? A : 0)) * V;
    const int c0 = c * chunk, c1 = min(V, c0 + chunk);
    u128 running = base;
    if (threadIdx.x == 0) s_mode = -1;
    for (int s0 = c0; s0 < c1; s0 += kSub) {
        const int v0 = s0 + threadIdx.x * 8;
        u128 w[8];
        float fp[8], fq[8];
        load8<VEC>(prow, v0, c1, fp);
        if (residual) load8<VEC>(qrow, v0, c1, fq);
        u128 tsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint64_t Ep = fixed_weight(fp[i], mp);
            if (residual) {
                uint64_t Eq = fixed_weight(fq[i], mq);
                u128 a = (u128)Ep * Sq, cc = (u128)Eq * Sp;
                w[i] = a > cc ? a - cc : (u128)0;
            } else {
                w[i] = Ep;
            }
            tsum += w[i];
        }
        u128 tinc = block_scan_u128(tsum, buf);
        u128 total = buf[kThreads - 1];
        u128 texc = running + tinc - tsum;
        if (running + tinc > T && texc <= T) {
            u128 cum = texc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cum += w[i];
                if (cum > T) {
                    s_mode = v0 + i;
                    break;
                }
            }
        }
        __syncthreads();
        if (s_mode >= 0) break;
        running += total;
    }
    if (threadIdx.x == 0) out[(size_t)b * (gamma + 1) + A] = s_mode >= 0 ? s_mode : c1 - 1;
}

// -------------------------------------------------------------------------
// draft-side sampling: the rows are Q[b] (B rows, gamma = 0 in the row
// kernels above, A_b = 0 so the draw kernel draws from the row's own E)
// -------------------------------------------------------------------------
// grid (b, chunk): this chunk's sum of E_v and its part of the entropy sum
// sum_v p_v log(p_v + 1e-9) (p_v = E_v / S in fp32); A_b = 0 for the draw.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) draft_chunk_kernel(const uint16_t *__restrict__ Q, int V, int chunk,
                                                               const uint32_t *__restrict__ maxenc,
                                                               const unsigned long long *__restrict__ sums,
                                                               unsigned long long *__restrict__ esum,
                                                               float *__restrict__ hpart,
                                                               int32_t *__restrict__ accbuf) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ unsigned long long she[kThreads / 32];
    __shared__ float shh[kThreads / 32];
    const int b = blockIdx.x, n_chunks = gridDim.y;
    const uint64_t S = sums[b];
    const float m = from_ordered_bits(maxenc[b]);
    const float inv = S ? (float)(1.0 / (double)S) : 0.0f;
    const uint16_t *row = Q + (size_t)b * V;
    const int c0 = blockIdx.y * chunk, c1 = min(V, c0 + chunk);
    unsigned long long e = 0;
    float h = 0.0f;
    if (S) {                                   // a row without mass has no weights
        for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += kSub) {
            float f[8];
            load8<VEC>(row, v0, c1, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t E = fixed_weight(f[i], m);
                const float p = (float)E * inv;
                e += E;
                h += p * logf(p + 1e-9f);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        e += __shfl_xor_sync(0xffffffffu, e, o);
        h += __shfl_xor_sync(0xffffffffu, h, o);
    }
    if ((threadIdx.x & 31) == 0) {
        she[threadIdx.x >> 5] = e;
        shh[threadIdx.x >> 5] = h;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long et = 0;
        float ht = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) {
            et += she[w];
            ht += shh[w];
        }
        esum[(size_t)b * n_chunks + blockIdx.y] = et;
        hpart[(size_t)b * n_chunks + blockIdx.y] = ht;
        if (blockIdx.y == 0) accbuf[b] = 0;
    }
}

// one thread per row: entropy from the chunk parts (in chunk order) and the
// confidence max_v E_v / S (the row maximum's weight, rint(qexp(0) 2^32))
__global__ void draft_features_kernel(int B, int n_chunks, const uint32_t *__restrict__ maxenc,
                                      const unsigned long long *__restrict__ sums,
                                      const float *__restrict__ hpart, float *__restrict__ confidence,
                                      float *__restrict__ entropy) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const uint64_t S = sums[b];
    float h = 0.0f;
    for (int c = 0; c < n_chunks; ++c) h += hpart[(size_t)b * n_chunks + c];
    entropy[b] = -h;
    const float m = from_ordered_bits(maxenc[b]);
    confidence[b] = S ? (float)((double)fixed_weight(m, m) / (double)S) : 0.0f;
}

// One launch per draft position: a cluster of C = 16 CTAs of NT threads per
// row (where the device schedules clusters of 16), CTA r over the
// slice [r span, (r + 1) span) of the row (span a multiple of 8).  Each
// thread loads its pieces of the slice once (all loads in flight together)
// and keeps them in registers: the maximum, then E_v, their sum, and E_v
// kept in shared memory (8 span bytes); from those, the entropy part and, in
// the one CTA whose slice holds the threshold, the draw.  Between the passes every CTA reads
// the others' partial results out of their shared memory.  The sums are the
// same integers as in the chunked kernels, so tokens and confidences are the
// same bits; the entropy's fp32 parts are added per slice.
constexpr int kDraftClusterMinV = 2048;
constexpr int kDraftThreads = 256;
constexpr int kDraftCacheMax = 200 * 1024;   // bytes of E_v one CTA keeps (its slice, 8 bytes each)
constexpr int kDraftIt = 6;                  // 8-logit pieces a thread holds (span <= kDraftIt * 8 NT)

// inclusive scan of one uint64 per thread over the block (warp shuffles,
// then the warps' totals in order); `total` gets the block's sum
template <int NT>
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long *wsum,
                                                             unsigned long long &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    unsigned long long off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const unsigned long long t = wsum[w];
        off += w < warp ? t : 0ull;
        tot += t;
    }
    __syncthreads();                           // wsum is free again
    total = tot;
    return v + off;
}

struct __align__(16) DraftPart {
    uint32_t maxe;              // the slice's largest logit, ordered bits
    float h;                    // the slice's sum of p log(p + 1e-9)
    unsigned long long sum;     // the slice's sum of E_v
};

template <bool VEC, int C, int NT>
__global__ void __launch_bounds__(NT) draft_cluster_kernel(const uint16_t *__restrict__ Q, int V, int span,
                                                                 uint64_t seed, uint64_t round, uint32_t slot,
                                                                 int32_t *__restrict__ token,
                                                                 float *__restrict__ confidence,
                                                                 float *__restrict__ entropy, int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) unsigned long long ecache[];   // E_v of the slice, v - c0
    __shared__ DraftPart part;
    __shared__ uint32_t shm[NT / 32];
    __shared__ unsigned long long shs[NT / 32];
    __shared__ float shh[NT / 32];
    __shared__ float s_m;
    __shared__ unsigned long long s_S, s_base, s_own;
    __shared__ int s_tok;
    const uint32_t r = umma::cluster_rank();
    const int b = blockIdx.y;
    const uint16_t *row = Q + (size_t)b * V;
    const int c0 = min(V, (int)r * span), c1 = min(V, c0 + span);

    // this thread's pieces: logits v0(it) .. v0(it) + 7, bf16 bits, -inf
    // past the slice
    uint4 raw[kDraftIt];
#pragma unroll
    for (int it = 0; it < kDraftIt; ++it) {
        const int v0 = c0 + (it * NT + (int)threadIdx.x) * 8;
        if (VEC && v0 + 8 <= c1) {
            raw[it] = __ldg(reinterpret_cast<const uint4 *>(row + v0));
        } else {
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = v0 + i < c1 ? (uint32_t)row[v0 + i] : 0xFF80u;
            raw[it] = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
        }
    }
    auto unpack = [](const uint4 &u, float (&f)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    };

    // the row maximum (NaN and +inf flagged, as in the row statistics)
    float m = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kDraftIt; ++it) {
        float f[8];
        unpack(raw[it], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bad |= isnan(f[i]) || f[i] == INFINITY;
            m = fmaxf(m, f[i]);
        }
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
    const uint32_t me = block_reduce_max<uint32_t, NT>(ordered_bits(m), shm);
    if (threadIdx.x == 0) part.maxe = me;
    umma::cluster_sync();
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {                    // lane q reads CTA q's part: one round trip
        uint32_t mx = lane < C ? umma::ld_peer_v4(&part, (uint32_t)lane).x : 0u;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_m = from_ordered_bits(mx);
    }
    __syncthreads();
    const float mrow = s_m;
    if (mrow == -INFINITY && r == 0 && threadIdx.x == 0) flag(st, QSPEC_ERR_NONFINITE);   // no mass

    // S = sum of E_v, and the sum of the slices before this one
    unsigned long long s = 0;
    if (mrow != -INFINITY)
#pragma unroll
        for (int it = 0; it < kDraftIt; ++it) {
            const int v0 = c0 + (it * NT + (int)threadIdx.x) * 8;
            if (v0 >= c1) break;
            float f[8];
            unpack(raw[it], f);
            unsigned long long E[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                E[i] = fixed_weight(f[i], mrow);   // 0 past the slice (-inf)
                s += E[i];
            }
            ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(ecache + (v0 - c0));
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_ulonglong2(E[2 * i], E[2 * i + 1]);
        }
    s = block_reduce_sum<NT>(s, shs);
    if (threadIdx.x == 0) part.sum = s;
    umma::cluster_sync();
    if (threadIdx.x < 32) {
        unsigned long long sq = 0;
        if (lane < C) {
            const uint4 w = umma::ld_peer_v4(&part, (uint32_t)lane);
            sq = (unsigned long long)w.z | ((unsigned long long)w.w << 32);
        }
        unsigned long long S = sq, below = lane < (int)r ? sq : 0ull;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            S += __shfl_xor_sync(0xffffffffu, S, o);
            below += __shfl_xor_sync(0xffffffffu, below, o);
        }
        if (lane == 0) {
            s_S = S;
            s_base = below;
            s_own = s;                         // thread 0 holds the block's sum
        }
    }
    __syncthreads();
    const unsigned long long S = s_S;

    // the slice's entropy part, p_v = E_v / S in fp32
    const float inv = S ? (float)(1.0 / (double)S) : 0.0f;
    float h = 0.0f;
    if (S)
        for (int v0 = c0 + threadIdx.x * 8; v0 < c1; v0 += NT * 8) {
            const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(ecache + (v0 - c0));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const ulonglong2 e2 = src[i >> 1];
                const unsigned long long E = i & 1 ? e2.y : e2.x;
                // E <= 2^32: through 32 bits, the same rounding
                const float Ef = E >> 32 ? 4294967296.0f : __uint2float_rn((uint32_t)E);
                const float p = Ef * inv;
                h += p * logf(p + 1e-9f);
            }
        }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if ((threadIdx.x & 31) == 0) shh[threadIdx.x >> 5] = h;
    __syncthreads();
    if (threadIdx.x == 0) {
        float ht = 0.0f;
        for (int w = 0; w < NT / 32; ++w) ht += shh[w];
        part.h = ht;
    }

    // the draw: v* = min{v : sum_{u<=v} E_u > T}, T = floor(U S / 2^24), in
    // the slice whose range of prefix sums holds T (every prefix sum is below
    // S < V 2^33, so 64 bits hold them)
    const unsigned long long T =
        (unsigned long long)(((u128)uniform24(seed, round, slot, (uint32_t)b) * S) >> 24);
    const unsigned long long base = s_base, own = s_own;
    if (S != 0 && base <= T && T - base < own) {
        if (threadIdx.x == 0) s_tok = -1;
        __syncthreads();
        unsigned long long running = base;
        for (int s0 = c0; s0 < c1; s0 += NT * 8) {
            const int v0 = s0 + threadIdx.x * 8;
            unsigned long long w[8];
            unsigned long long tsum = 0;
            if (v0 < c1) {
                const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(ecache + (v0 - c0));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const ulonglong2 e2 = src[i];
                    w[2 * i] = e2.x;
                    w[2 * i + 1] = e2.y;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = 0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) tsum += w[i];
            unsigned long long total;
            const unsigned long long tinc = block_scan_u64<NT>(tsum, shs, total);
            const unsigned long long texc = running + tinc - tsum;
            if (running + tinc > T && texc <= T) {
                unsigned long long cum = texc;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cum += w[i];
                    if (cum > T) {
                        s_tok = v0 + i;
                        break;
                    }
                }
            }
            __syncthreads();
            if (s_tok >= 0) break;
            running += total;
        }
        if (threadIdx.x == 0) token[b] = s_tok >= 0 ? s_tok : c1 - 1;
    } else if (S == 0 && r == C - 1 && threadIdx.x == 0) {
        token[b] = V - 1;                      // a row without mass (flagged above)
    }

    // the features: entropy from the slices' parts (a fixed shuffle tree),
    // the confidence max_v E_v / S as in the chunked path
    umma::cluster_sync();
    if (r == 0 && threadIdx.x < 32) {
        float ht = lane < C ? umma::ld_peer_f32(&part.h, (uint32_t)lane) : 0.0f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ht += __shfl_xor_sync(0xffffffffu, ht, o);
        if (lane == 0) {
            entropy[b] = -ht;
            confidence[b] = S ? (float)((double)fixed_weight(mrow, mrow) / (double)S) : 0.0f;
        }
    }
    umma::cluster_sync();                      // every CTA's shared memory stays until CTA 0 has read it
}

}  // namespace

}  // namespace qspec

using namespace qspec;

extern "C" size_t qspec_verify_workspace_bytes(int B, int gamma, int V) {
    if (B < 1 || gamma < 1 || gamma > QSPEC_MAX_GAMMA || V < 1) return 0;
    return make_layout(B, gamma, V).total;
}

static int verify_args(const void *p, const int32_t *draft, int B, int gamma, int V, const int32_t *n_acc,
                       const int32_t *out, const void *ws, size_t ws_bytes) {
    if (!p || !draft || !n_acc || !out || !ws) return QSPEC_ERR_NULL;
    if (B < 1 || gamma < 1 || gamma > QSPEC_MAX_GAMMA || V < 1) return QSPEC_ERR_SHAPE;
    if (!aligned(p, 2) || !aligned(draft, 4) || !aligned(n_acc, 4) || !aligned(out, 4) ||
        !aligned(ws, 16))
        return QSPEC_ERR_ALIGN;
    if (ws_bytes < make_layout(B, gamma, V).total) return QSPEC_ERR_WORKSPACE;
    return QSPEC_OK;
}

extern "C" int qspec_verify_greedy(const uint16_t *p_logits, const int32_t *draft, int B, int gamma,
                                   int V, int32_t *n_acc, int32_t *out, void *workspace,
                                   size_t ws_bytes, int32_t *dev_status, qspec_stream_t stream) {
    int rc = verify_args(p_logits, draft, B, gamma, V, n_acc, out, workspace, ws_bytes);
    if (rc) return rc;
    rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    Layout L = make_layout(B, gamma, V);
    char *ws = static_cast<char *>(workspace);
    auto *keys = reinterpret_cast<unsigned long long *>(ws + L.off_key);
    const int rows = B * (gamma + 1);
    bool vec = (V % 8 == 0) && aligned(p_logits, 16);
    // one CTA per row when there are at least two rows per SM, else each row
    // split into chunks so that the grid covers about two CTAs per SM; one
    // key per (row, chunk), no atomics and no clearing
    const int target = 2 * sm_count();
    int nch = rows >= target ? 1 : std::min(kMaxChunks, (target + rows - 1) / rows);
    const int subs = (V + kSub - 1) / kSub;
    const int chunk = ((subs + nch - 1) / nch) * kSub;
    nch = (V + chunk - 1) / chunk;
    if ((size_t)rows * nch > (size_t)rows + kGreedyExtraKeys) return QSPEC_ERR_UNSUPPORTED;
    dim3 grid((unsigned)rows, (unsigned)nch);
    rc = vec ? launch_pdl("qspec_verify_greedy", greedy_argmax_kernel<true>, grid, dim3(kThreads), 0, st, p_logits,
                          V, chunk, keys, dev_status)
             : launch_pdl("qspec_verify_greedy", greedy_argmax_kernel<false>, grid, dim3(kThreads), 0, st, p_logits,
                          V, chunk, keys, dev_status);
    if (rc) return rc;
    return launch_pdl("qspec_verify_greedy", greedy_finalize_kernel, dim3((B + 127) / 128), dim3(128), 0, st,
                      keys, nch, draft, B, gamma, V, n_acc, out, dev_status);
}

template <bool VEC>
static int launch_sample(const uint16_t *P, const uint16_t *Q, const int32_t *draft, int B, int gamma,
                          int V, uint64_t seed, uint64_t round, int32_t *n_acc, int32_t *out,
                          const Layout &L, char *ws, int32_t *dev_status, cudaStream_t st) {
    auto *maxenc = reinterpret_cast<uint32_t *>(ws + L.off_max);
    auto *sums = reinterpret_cast<unsigned long long *>(ws + L.off_sum);
    auto *rsum = reinterpret_cast<u128 *>(ws + L.off_rsum);
    auto *esum = reinterpret_cast<unsigned long long *>(ws + L.off_esum);
    auto *accbuf = reinterpret_cast<int32_t *>(ws + L.off_acc);
    const int rows = B * (2 * gamma + 1);
    const char *w = "qspec_verify_sample";
    int rc;
    if (rows >= 2 * sm_count()) {
        // enough rows: one CTA per row, both statistics in one launch
        rc = launch_pdl(w, sample_rowstats_kernel<VEC>, dim3(rows), dim3(kRowThreads), 0, st, P, Q, B, gamma, V,
                        maxenc, sums, dev_status);
        if (rc) return rc;
    } else {
        // few rows: chunks of every row; maxima and sums combined with atomics
        // from 0 (below every encoded value)
        cudaError_t e = cudaMemsetAsync(ws + L.off_max, 0, L.off_rsum - L.off_max, st);
        if (e != cudaSuccess) {
            set_last_error("qspec_verify_sample memset", e);
            return QSPEC_ERR_LAUNCH;
        }
        dim3 grid_rows((unsigned)rows, (unsigned)L.n_chunks);
        rc = launch_pdl(w, sample_rowmax_kernel<VEC>, grid_rows, dim3(kThreads), 0, st, P, Q, B, gamma, V, L.chunk,
                        maxenc, dev_status);
        if (rc) return rc;
        rc = launch_pdl(w, sample_rowsum_kernel<VEC>, grid_rows, dim3(kThreads), 0, st, P, Q, B, gamma, V,
                        L.chunk, maxenc, sums, dev_status);
        if (rc) return rc;
    }
    dim3 grid_seq((unsigned)B, (unsigned)L.n_chunks);
    rc = launch_pdl(w, sample_residual_kernel<VEC>, grid_seq, dim3(kThreads), 0, st, P, Q, draft, B, gamma, V,
                    L.chunk, seed, round, maxenc, sums, rsum, esum, accbuf, n_acc, out, dev_status);
    if (rc) return rc;
    return launch_pdl(w, sample_draw_kernel<VEC>, dim3(B), dim3(kThreads), 0, st, P, Q, B, gamma, V, L.chunk,
                      L.n_chunks, seed, round, (uint32_t)gamma, maxenc, sums, rsum, esum, accbuf, out);
}

extern "C" int qspec_verify_sample(const uint16_t *p_logits, const uint16_t *q_logits,
                                   const int32_t *draft, int B, int gamma, int V, uint64_t seed,
                                   uint64_t round, int32_t *n_acc, int32_t *out, void *workspace,
                                   size_t ws_bytes, int32_t *dev_status, qspec_stream_t stream) {
    if (!q_logits) return QSPEC_ERR_NULL;
    int rc = verify_args(p_logits, draft, B, gamma, V, n_acc, out, workspace, ws_bytes);
    if (rc) return rc;
    if (!aligned(q_logits, 2)) return QSPEC_ERR_ALIGN;
    rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    Layout L = make_layout(B, gamma, V);
    char *ws = static_cast<char *>(workspace);
    bool vec = (V % 8 == 0) && aligned(p_logits, 16) && aligned(q_logits, 16);
    return vec ? launch_sample<true>(p_logits, q_logits, draft, B, gamma, V, seed, round, n_acc, out, L, ws,
                                     dev_status, st)
               : launch_sample<false>(p_logits, q_logits, draft, B, gamma, V, seed, round, n_acc, out, L, ws,
                                      dev_status, st);
}

// ---------------------------------------------------------------------------
// Sampled verification without any allocation by the caller.
//
// Some callers cannot call cudaMalloc at all: code running inside a CUDA
// graph that is being captured (where allocation is not a stream operation),
// plugins that own no allocator, or runtimes whose memory is fully reserved
// up front.  For them this variant keeps its scratch in a fixed device array
// that is part of the library image: every GPU that loads the library holds
// QSPEC_VERIFY_NOALLOC_SCRATCH_BYTES of it until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[QSPEC_VERIFY_NOALLOC_SCRATCH_BYTES];

// Device address of the array, looked up with the device current and
// remembered per CUDA context (keyed on the context's unique id, so a
// cudaDeviceReset or a new context on the same device triggers a fresh
// lookup instead of handing the kernels an address from a context that no
// longer exists).  In host code the symbol g_noalloc_scratch is only a
// host-side stand-in; a kernel handed it would read the wrong memory.
namespace {

typedef CUresult (*CtxGetCurrent)(CUcontext *);
typedef CUresult (*CtxGetId)(CUcontext, unsigned long long *);

struct NoallocSlot {
    unsigned long long ctx_id;
    void *addr;
};
NoallocSlot g_noalloc_slot[64];
std::mutex g_noalloc_mu;

// id of the calling thread's current context; false when there is none or
// the driver entry points are not available
bool current_ctx_id(unsigned long long *id) {
    static CtxGetCurrent get_current = nullptr;
    static CtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetId>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
    return get_id(c, id) == CUDA_SUCCESS;
}

}  // namespace

static int noalloc_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice", e);
        return QSPEC_ERR_LAUNCH;
    }
    if (dev < 0 || dev >= 64) return QSPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    NoallocSlot &slot = g_noalloc_slot[dev];
    if (have_id && slot.addr != nullptr && slot.ctx_id == id) {
        *ptr = slot.addr;
        return QSPEC_OK;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        set_last_error("cudaGetSymbolAddress(g_noalloc_scratch)", e);
        return QSPEC_ERR_LAUNCH;
    }
    // the lookup makes the device's primary context current if none was;
    // remember the address only when the context can be identified
    if (current_ctx_id(&id)) {
        slot.ctx_id = id;
        slot.addr = p;
    } else {
        slot.addr = nullptr;
    }
    *ptr = p;
    return QSPEC_OK;
}

extern "C" int qspec_verify_sample_noalloc(const uint16_t *p_logits, const uint16_t *q_logits,
                                           const int32_t *draft, int B, int gamma, int V, uint64_t seed,
                                           uint64_t round, int32_t *n_acc, int32_t *out,
                                           int32_t *dev_status, qspec_stream_t stream) {
    if (!p_logits || !q_logits || !draft || !n_acc || !out) return QSPEC_ERR_NULL;
    if (B < 1 || gamma < 1 || gamma > QSPEC_MAX_GAMMA || V < 1) return QSPEC_ERR_SHAPE;
    if (make_layout(B, gamma, V).total > (size_t)QSPEC_VERIFY_NOALLOC_SCRATCH_BYTES)
        return QSPEC_ERR_WORKSPACE;
    int rc = check_device();
    if (rc) return rc;
    void *scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return qspec_verify_sample(p_logits, q_logits, draft, B, gamma, V, seed, round, n_acc, out, scratch,
                               QSPEC_VERIFY_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Draft-side sampling with the draft statistics: the row statistics of the
// sampled verification over the B draft rows (gamma = 0), per-chunk weight
// sums and entropy parts, the draw of the verification's bonus path with the
// uniform of slot 16 + step, then the features.  The workspace is the
// verification layout for gamma = 0; the residual chunk sums (unused here)
// hold the entropy parts.
// ---------------------------------------------------------------------------
extern "C" size_t qspec_draft_workspace_bytes(int B, int V) {
    if (B < 1 || V < 1) return 0;
    return make_layout(B, 0, V).total;
}

// 16 when clusters of 16 CTAs (a size above the portable 8) can be
// scheduled for the draft kernel on this device, else 0 (the chunked path
// then runs); settled once per device (both instances get the attribute),
// before any capture
static int draft_cluster_size() {
    static std::mutex mu;
    static int known[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (known[dev] == 0) {
        const void *k1 = reinterpret_cast<const void *>(draft_cluster_kernel<true, 16, kDraftThreads>);
        const void *k0 = reinterpret_cast<const void *>(draft_cluster_kernel<false, 16, kDraftThreads>);
        int c = -1;
        if (cudaFuncSetAttribute(k1, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
            cudaFuncSetAttribute(k0, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
            smem_limit_once(k1, kDraftCacheMax) == QSPEC_OK && smem_limit_once(k0, kDraftCacheMax) == QSPEC_OK) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16, 1);
            cfg.blockDim = dim3(kDraftThreads);
            cfg.dynamicSmemBytes = kDraftCacheMax;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 16;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n0 = 0, n1 = 0;
            if (cudaOccupancyMaxActiveClusters(&n1, k1, &cfg) == cudaSuccess && n1 >= 1 &&
                cudaOccupancyMaxActiveClusters(&n0, k0, &cfg) == cudaSuccess && n0 >= 1)
                c = 16;
        }
        cudaGetLastError();                    // a refused size leaves no error behind
        known[dev] = c;
    }
    return known[dev] > 0 ? known[dev] : 0;
}

template <bool VEC>
static int launch_draft(const uint16_t *Q, int B, int V, uint64_t seed, uint64_t round, int step, int32_t *token,
                        float *confidence, float *entropy, const Layout &L, char *ws, int32_t *dev_status,
                        cudaStream_t st) {
    auto *maxenc = reinterpret_cast<uint32_t *>(ws + L.off_max);
    auto *sums = reinterpret_cast<unsigned long long *>(ws + L.off_sum);
    auto *rsum = reinterpret_cast<u128 *>(ws + L.off_rsum);
    auto *hpart = reinterpret_cast<float *>(ws + L.off_rsum);
    auto *esum = reinterpret_cast<unsigned long long *>(ws + L.off_esum);
    auto *accbuf = reinterpret_cast<int32_t *>(ws + L.off_acc);
    const char *w = "qspec_draft_sample";
    int rc;
    const int C = B < 2 * sm_count() && V >= kDraftClusterMinV ? draft_cluster_size() : 0;
    const int span = C ? ((V + C - 1) / C + 7) / 8 * 8 : 0;
    if (C == 16 && (size_t)span * 8 <= (size_t)kDraftCacheMax && span <= kDraftIt * 8 * kDraftThreads) {
        const uint32_t slot = (uint32_t)(QSPEC_MAX_GAMMA + step);
        const size_t smem = (size_t)span * 8;
        return launch_pdl_cluster(w, draft_cluster_kernel<VEC, 16, kDraftThreads>, dim3(16, (unsigned)B),
                                  dim3(kDraftThreads), smem, st, 16, Q, V, span, seed, round, slot, token, confidence,
                                  entropy, dev_status);
    }
    if (B >= 2 * sm_count()) {
        rc = launch_pdl(w, sample_rowstats_kernel<VEC>, dim3(B), dim3(kRowThreads), 0, st, Q, Q, B, 0, V, maxenc,
                        sums, dev_status);
        if (rc) return rc;
    } else {
        cudaError_t e = cudaMemsetAsync(ws + L.off_max, 0, L.off_rsum - L.off_max, st);
        if (e != cudaSuccess) {
            set_last_error("qspec_draft_sample memset", e);
            return QSPEC_ERR_LAUNCH;
        }
        dim3 grid_rows((unsigned)B, (unsigned)L.n_chunks);
        rc = launch_pdl(w, sample_rowmax_kernel<VEC>, grid_rows, dim3(kThreads), 0, st, Q, Q, B, 0, V, L.chunk,
                        maxenc, dev_status);
        if (rc) return rc;
        rc = launch_pdl(w, sample_rowsum_kernel<VEC>, grid_rows, dim3(kThreads), 0, st, Q, Q, B, 0, V, L.chunk,
                        maxenc, sums, dev_status);
        if (rc) return rc;
    }
    rc = launch_pdl(w, draft_chunk_kernel<VEC>, dim3((unsigned)B, (unsigned)L.n_chunks), dim3(kThreads), 0, st, Q, V,
                    L.chunk, maxenc, sums, esum, hpart, accbuf);
    if (rc) return rc;
    rc = launch_pdl(w, sample_draw_kernel<VEC>, dim3(B), dim3(kThreads), 0, st, Q, Q, B, 0, V, L.chunk, L.n_chunks,
                    seed, round, (uint32_t)(QSPEC_MAX_GAMMA + step), maxenc, sums, rsum, esum, accbuf, token);
    if (rc) return rc;
    return launch_pdl(w, draft_features_kernel, dim3((B + 127) / 128), dim3(128), 0, st, B, L.n_chunks, maxenc, sums,
                      hpart, confidence, entropy);
}

extern "C" int qspec_draft_sample(const uint16_t *q_logits, int B, int V, uint64_t seed, uint64_t round, int step,
                                  int32_t *token, float *confidence, float *entropy, void *workspace,
                                  size_t ws_bytes, int32_t *dev_status, qspec_stream_t stream) {
    if (!q_logits || !token || !confidence || !entropy || !workspace) return QSPEC_ERR_NULL;
    if (B < 1 || V < 1 || step < 1 || step > QSPEC_MAX_GAMMA) return QSPEC_ERR_SHAPE;
    if (!aligned(q_logits, 2) || !aligned(token, 4) || !aligned(confidence, 4) || !aligned(entropy, 4) ||
        !aligned(workspace, 16))
        return QSPEC_ERR_ALIGN;
    const Layout L = make_layout(B, 0, V);
    if (ws_bytes < L.total) return QSPEC_ERR_WORKSPACE;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    char *ws = static_cast<char *>(workspace);
    const bool vec = (V % 8 == 0) && aligned(q_logits, 16);
    return vec ? launch_draft<true>(q_logits, B, V, seed, round, step, token, confidence, entropy, L, ws, dev_status,
                                    st)
               : launch_draft<false>(q_logits, B, V, seed, round, step, token, confidence, entropy, L, ws,
                                     dev_status, st);
}
