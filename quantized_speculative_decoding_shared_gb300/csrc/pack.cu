// pack.cu -- a1: pack INT4 weight codes two per byte and interleave the fp16
// group scale and zero point into one 32-bit word per (row, group).
//
// QSPEC summary page, background terms: W^ = s (W_INT4 - z); "QSPEC
// structure": one 4-bit weight set serves both the W4A4 and W4A16 kernels.
// HBM-bound bit moves: 1 byte read per code, half a byte written.
#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

// One thread per 32 codes: two 16-byte loads, one 16-byte store.
__global__ void __launch_bounds__(256) pack_codes_kernel(const uint4 *__restrict__ codes,
                                                        size_t n_chunks, uint4 *__restrict__ packed,
                                                        int32_t *st) {
    bool bad = false;
    for (size_t c = blockIdx.x * (size_t)blockDim.x + threadIdx.x; c < n_chunks;
         c += (size_t)gridDim.x * blockDim.x) {
        uint4 a = __ldcs(codes + 2 * c), b = __ldcs(codes + 2 * c + 1);
        uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w0 = in[2 * i], w1 = in[2 * i + 1];
            bad |= ((w0 | w1) & 0xF0F0F0F0u) != 0;
            // bytes (c0 c1 c2 c3): c0 | c1 << 4 lands in byte 0, c2 | c3 << 4 in byte 2
            uint32_t t0 = (w0 | (w0 >> 4)) & 0x00FF00FFu;
            uint32_t t1 = (w1 | (w1 >> 4)) & 0x00FF00FFu;
            out[i] = __byte_perm(t0, t1, 0x6420);
        }
        __stcs(packed + c, make_uint4(out[0], out[1], out[2], out[3]));
    }
    if (bad) flag(st, QSPEC_ERR_RANGE);
}

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint16_t *__restrict__ s,
                                                         const uint16_t *__restrict__ z, size_t n,
                                                         uint32_t *__restrict__ sz, int32_t *st) {
    int err = QSPEC_OK;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        uint16_t sb = s[i], zb = z[i];
        if ((sb & 0x7C00u) == 0x7C00u) err = QSPEC_ERR_NONFINITE;
        float zv = __half2float(__ushort_as_half(zb));
        if (!(zv >= 0.0f && zv <= 15.0f && zv == floorf(zv))) err = err ? err : QSPEC_ERR_ZERO_POINT;
        sz[i] = (uint32_t)sb | ((uint32_t)zb << 16);
    }
    if (err) flag(st, err);
}

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_pack_weights(const uint8_t *codes, const uint16_t *s_fp16,
                                  const uint16_t *z_fp16, int N, int K, uint8_t *packed,
                                  uint32_t *sz, int32_t *dev_status, qspec_stream_t stream) {
    if (!codes || !s_fp16 || !z_fp16 || !packed || !sz) return QSPEC_ERR_NULL;
    if (N < 1 || K < kGroup || K % kGroup) return QSPEC_ERR_SHAPE;
    if (!aligned(codes, 16) || !aligned(packed, 16) || !aligned(sz, 4) || !aligned(s_fp16, 2) ||
        !aligned(z_fp16, 2))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    size_t n_chunks = (size_t)N * K / 32;
    size_t n_groups = (size_t)N * (K / kGroup);
    int sms = sm_count();
    unsigned g1 = (unsigned)std::min<size_t>((n_chunks + 255) / 256, (size_t)sms * 8);
    unsigned g2 = (unsigned)std::min<size_t>((n_groups + 255) / 256, (size_t)sms * 8);
    pack_codes_kernel<<<g1, 256, 0, st>>>(reinterpret_cast<const uint4 *>(codes), n_chunks,
                                          reinterpret_cast<uint4 *>(packed), dev_status);
    pack_scales_kernel<<<g2, 256, 0, st>>>(s_fp16, z_fp16, n_groups, sz, dev_status);
    const int lrc = check_launch("qspec_pack_weights");
    if (lrc == QSPEC_OK) {
        count_launch();
        count_launch();
    }
    return lrc;
}
