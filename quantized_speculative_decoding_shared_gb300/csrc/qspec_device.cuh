// qspec_device.cuh -- device helpers shared by the library's kernels.
//
// Nothing here is shared with the CPU oracle: the Philox generator and the
// fixed-point exp are written separately on each side from their published
// definitions.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qspec.h"

namespace qspec {

constexpr int kGroup = QSPEC_GROUP;

// Programmatic dependent launch (PDL).  A kernel launched with
// launch_pdl() may start while the previous kernel in the stream is still
// running.  Rule kept by every kernel of this library: before pdl_wait() it
// only reads immutable data (packed weights, scale/zero words); every read
// of another kernel's output and every write comes after pdl_wait(), which
// returns once the previous grid has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next PDL-launched kernel be scheduled as this grid's CTAs retire.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// First data error wins: later codes never overwrite an earlier one.
__device__ __forceinline__ void flag(int32_t *st, int code) {
    if (st != nullptr && code != QSPEC_OK) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
    return __uint_as_float(b << 16);
}

// fp32 -> bf16 bits, round to nearest even (the bf16 intrinsic).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Monotone map of fp32 onto uint32: a < b (as floats, no NaN) iff enc(a) < enc(b).
// enc(x) > 0 for every x, so 0 works as a "minus infinity" start value.
__device__ __forceinline__ uint32_t ordered_bits(float x) {
    uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t e) {
    uint32_t u = (e & 0x80000000u) ? (e & 0x7fffffffu) : ~e;
    return __uint_as_float(u);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
// published multipliers, key bumped by the published Weyl constants.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
        uint32_t hi0 = __umulhi(m0, c0), lo0 = m0 * c0;
        uint32_t hi1 = __umulhi(m1, c2), lo1 = m1 * c2;
        uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// 24-bit uniform for draw `slot` of sequence b in verification round `round`.
__device__ __forceinline__ uint32_t uniform24(uint64_t seed, uint64_t round, uint32_t slot,
                                              uint32_t b) {
    return philox_word0(slot, b, (uint32_t)round, (uint32_t)(round >> 32), (uint32_t)seed,
                        (uint32_t)(seed >> 32)) >> 8;
}

// ---------------------------------------------------------------------------
// Fixed-point softmax weight E = rint(e^(l - m) * 2^32), l <= m.
// e^x for x in [-32, 0]: Cody-Waite reduction x = n ln2 + r (ln2 split into a
// 12-significant-bit head and a tail), degree-7 Taylor polynomial of e^r in
// Horner form, exact scaling by 2^n.  Every step is one fp32 operation,
// rounded to nearest; the fused steps are explicit fmas.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float qexp(float x) {
    if (x < -32.0f) return 0.0f;
    const float log2e = __uint_as_float(0x3FB8AA3Bu);
    const float ln2_hi = __uint_as_float(0x3F317200u);
    const float ln2_lo = __uint_as_float(0x35BFBE8Eu);
    float n = rintf(__fmul_rn(x, log2e));
    float r = __fmaf_rn(-n, ln2_hi, x);
    r = __fmaf_rn(-n, ln2_lo, r);
    float p = __uint_as_float(0x39500D01u);            // 1/7!
    p = __fmaf_rn(p, r, __uint_as_float(0x3AB60B61u)); // 1/6!
    p = __fmaf_rn(p, r, __uint_as_float(0x3C088889u)); // 1/5!
    p = __fmaf_rn(p, r, __uint_as_float(0x3D2AAAABu)); // 1/4!
    p = __fmaf_rn(p, r, __uint_as_float(0x3E2AAAABu)); // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    int e = (int)n;                                     // -47 <= e <= 0
    return __fmul_rn(p, __int_as_float((e + 127) << 23));
}

// rint(qexp(l - m) * 2^32), computed with the same fp32 operations as
// qexp followed by the product, in fewer instructions:
//   - rint(x log2e) by adding and subtracting 1.5 * 2^23 (round to nearest
//     even, as rintf; exact for |x log2e| < 2^22), which also leaves n in the
//     low bits of the sum;
//   - p * 2^n * 2^32 as one product with 2^(n + 32): both scalings are exact
//     (p in [0.7, 1.5], n >= -47, so p 2^n is a normal number);
//   - the value is at most 2^32, and below it at most 2^32 - 256, so a 32-bit
//     conversion covers everything but the row maximum itself.
//   - no branch: below -32 the weight is 0, selected at the end (the
//     polynomial runs on -32 instead), so a thread's independent weights
//     interleave.
__device__ __forceinline__ uint64_t fixed_weight(float l, float m) {
    const float x0 = __fsub_rn(l, m);
    const float x = x0 < -32.0f ? -32.0f : x0;
    const float log2e = __uint_as_float(0x3FB8AA3Bu);
    const float ln2_hi = __uint_as_float(0x3F317200u);
    const float ln2_lo = __uint_as_float(0x35BFBE8Eu);
    const float t = __fadd_rn(__fmul_rn(x, log2e), 12582912.0f);
    const float n = __fsub_rn(t, 12582912.0f);
    float r = __fmaf_rn(-n, ln2_hi, x);
    r = __fmaf_rn(-n, ln2_lo, r);
    float p = __uint_as_float(0x39500D01u);            // 1/7!
    p = __fmaf_rn(p, r, __uint_as_float(0x3AB60B61u)); // 1/6!
    p = __fmaf_rn(p, r, __uint_as_float(0x3C088889u)); // 1/5!
    p = __fmaf_rn(p, r, __uint_as_float(0x3D2AAAABu)); // 1/4!
    p = __fmaf_rn(p, r, __uint_as_float(0x3E2AAAABu)); // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int e = (int)(__float_as_uint(t) - 0x4B400000u);   // n
    const float v = __fmul_rn(p, __int_as_float((e + 127 + 32) << 23));
    const uint64_t w = v >= 4294967296.0f ? (1ull << 32) : (uint64_t)__float2uint_rn(v);
    return x0 < -32.0f ? 0ull : w;
}

// Reciprocal of x within 1 ulp (the PTX rcp.approx instruction; subnormal x
// flushes to zero and gives inf).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}

// a2 quantisation of one 128-element group by 16 / kVec lanes, each with
// kVec 16-byte words of 8 bf16 (consecutive elements; the lanes of a group
// are consecutive and aligned, and every lane of the warp takes part, each
// group of lanes with its own group): amax over the group, sx = amax / 7
// (IEEE division), q = clamp(rint(x / sx), -7, 7) (0 when sx == 0), qs =
// sum q over the group.  nib[i] gets the codes of v[i] as nibbles (two's
// complement, code e in bits 4e..4e+3); `bad` is set by a NaN or inf input.
// Shared by the quantiser and the kernels that quantise their own
// activations, so all agree bit for bit.
//
// The quotient is taken as one Newton step from the approximate reciprocal
// y = rcp.approx(sx): q0 = x y, r = fma(-q0, sx, x) (the exact remainder),
// t = fma(r, y, q0).  For every pair of bf16 values with |x| <= amax and
// sx = amax / 7 >= 1e-30 (all 1.05e9 of them, checked exhaustively on the
// device against the IEEE division), rint(t) equals rint(x / sx) and lies
// in [-7, 7], so no clamp and no tie test are needed; groups with sx below
// 1e-30 take the IEEE division.  rint(t) is t + 1.5 * 2^23 rounded to
// nearest (even), whose low four bits are then the code; the sum of the
// rounded values is exact, and not finite exactly when some input is not (a
// NaN or inf x makes its t a NaN).
template <int kVec>
__device__ __forceinline__ void quant_group(const uint4 (&v)[kVec], float &scale, int &qsum, bool &bad,
                                            uint32_t (&nib)[kVec]) {
    static_assert(kVec == 1 || kVec == 2 || kVec == 4, "16, 8 or 4 lanes per group");
    constexpr float kMagic = 12582912.0f;                  // 1.5 * 2^23
    float f[kVec * 8];
#pragma unroll
    for (int c = 0; c < kVec; ++c) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
            f[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    // (maxima, sums and nibble packing as trees: short dependency chains)
    float a[kVec * 8];
#pragma unroll
    for (int i = 0; i < kVec * 8; ++i) a[i] = fabsf(f[i]);
#pragma unroll
    for (int w = kVec * 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) a[i] = fmaxf(a[i], a[i + w]);
    float amax = a[0];
#pragma unroll
    for (int o = 8 / kVec; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    scale = __fdiv_rn(amax, 7.0f);
    const bool tiny = scale < 1.0e-30f;                     // 0 included: then every x is 0
    const float y = tiny ? 0.0f : rcp_approx(scale);
    float r[kVec * 8];
    uint32_t e[kVec * 8];
#pragma unroll
    for (int i = 0; i < kVec * 8; ++i) {
        const float q0 = __fmul_rn(f[i], y);
        const float t = __fmaf_rn(__fmaf_rn(-q0, scale, f[i]), y, q0);
        const float m = __fadd_rn(t, kMagic);
        r[i] = __fsub_rn(m, kMagic);                          // rint(t)
        e[i] = (__float_as_uint(m) & 15u) << (4 * (i & 7));
    }
#pragma unroll
    for (int w = kVec * 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) r[i] = __fadd_rn(r[i], r[i + w]);   // integers: exact in any order
#pragma unroll
    for (int c = 0; c < kVec; ++c) {
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) e[8 * c + i] |= e[8 * c + i + w];
        nib[c] = e[8 * c];
    }
    const float qf = r[0];
    bad |= !isfinite(qf);
    int sum = (int)qf;
    const bool redo = tiny && scale != 0.0f;
    if (__any_sync(0xffffffffu, redo)) {                     // sx below 1e-30: the IEEE division
        if (redo) {
            sum = 0;
#pragma unroll
            for (int c = 0; c < kVec; ++c) {
                uint32_t n = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = max(-7, min(7, (int)rintf(__fdiv_rn(f[8 * c + i], scale))));
                    sum += q;
                    n |= (uint32_t)(q & 15) << (4 * i);
                }
                nib[c] = n;
            }
        }
    }
#pragma unroll
    for (int o = 8 / kVec; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    qsum = sum;
}

// The same by half a warp (16 lanes x one 16-byte word); returns the nibbles.
__device__ __forceinline__ uint32_t quant_group_halfwarp(uint4 v, float &scale, int &qsum, bool &bad) {
    const uint4 a[1] = {v};
    uint32_t n[1];
    quant_group<1>(a, scale, qsum, bad, n);
    return n[0];
}

// A W4A16 linear whose epilogue also writes its outputs into a KV cache
// (the verify pass's k / v projection, QSPEC summary page, "QSPEC
// structure": the accepted tokens' cache entries become the W4A16 ones).
// Output columns [c0, c0 + H D) are K and the next H D columns V (either
// cache may be null); output row m = b (gamma + 1) + r is position
// base[b] + r of sequence b in the caches [B][H][T][D], written for
// r <= nacc[b], or for every r when nacc is null.  A sequence with
// base[b] < 0, nacc[b] outside [0, gamma] or base[b] + (its last r) >= T is
// left untouched and QSPEC_ERR_RANGE is flagged.  k == v == null: no cache
// output.
struct KvOut {
    uint16_t *k, *v;
    const int32_t *base, *nacc;
    int c0, H, D, T, gamma;
    int32_t *st;
};

__device__ __forceinline__ void kv_store(const KvOut &kv, int m, int n, uint16_t val) {
    if (kv.k == nullptr && kv.v == nullptr) return;
    const int HD = kv.H * kv.D, j = n - kv.c0;
    if (j < 0 || j >= 2 * HD) return;
    uint16_t *cache = j < HD ? kv.k : kv.v;
    if (cache == nullptr) return;
    const int jj = j < HD ? j : j - HD, h = jj / kv.D, d = jj - h * kv.D;
    const int b = m / (kv.gamma + 1), r = m - b * (kv.gamma + 1);
    const int last = kv.nacc ? kv.nacc[b] : kv.gamma, p0 = kv.base[b];
    if (p0 < 0 || last < 0 || last > kv.gamma || p0 + last >= kv.T) {
        flag(kv.st, QSPEC_ERR_RANGE);
        return;
    }
    if (r > last) return;
    cache[(((size_t)b * kv.H + h) * kv.T + p0 + r) * kv.D + d] = val;
}

typedef unsigned __int128 u128;

}  // namespace qspec
