// actquant.cu -- a2: symmetric INT4 quantisation of bf16 activations per token
// and 128-group (QSPEC summary page, background terms: W4A4 quantises the
// activations to 4 bits as well as the weights).
//
// Per (m, g): amax = max |x|, sx = amax / 7 (IEEE fp32 division),
// q = clamp(rint(x / sx), -7, 7) (0 when sx == 0; the quotient through the
// rounded reciprocal, the division itself near rounding ties), qs = sum q.
// Eight lanes per group, four groups per warp: 8 lanes x 16 bf16 (two
// 16-byte loads each), amax and qs by shuffles over the eight lanes.
// HBM-bound: 2 bytes read and ~0.53 bytes written per element.
#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t *__restrict__ x, int M, int K,
                                                       int ldx, uint8_t *__restrict__ xq,
                                                       float *__restrict__ sx,
                                                       int32_t *__restrict__ qs, int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    const int G = K / kGroup;
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3, l8 = lane & 7;               // group of the quad, lane in the group
    const int qpr = (G + 3) / 4;                             // group quads per row
    const int tasks = M * qpr;                               // one quad per warp-task
    const int n_warps = (int)((gridDim.x * blockDim.x) >> 5);
    int w0 = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    bool bad = false;
    // kBatch quad-tasks per warp and pass, their loads issued first; (row,
    // quad) stepped by n_warps per task with one division per pass
    constexpr int kBatch = 2;
    for (; w0 < tasks; w0 += kBatch * n_warps) {
        uint4 v[kBatch][2];
        int mm[kBatch], gg[kBatch];
        int m = w0 / qpr, p = w0 - m * qpr;
        const int dm = n_warps / qpr, dp = n_warps - dm * qpr;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int g = 4 * p + sub;
            const bool active = m < M && g < G;
            mm[j] = active ? m : -1;
            gg[j] = g;
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)m * ldx + (size_t)g * kGroup) + 2 * l8;
            v[j][0] = active ? __ldcs(src) : make_uint4(0u, 0u, 0u, 0u);
            v[j][1] = active ? __ldcs(src + 1) : make_uint4(0u, 0u, 0u, 0u);
            m += dm;
            p += dp;
            if (p >= qpr) {
                p -= qpr;
                ++m;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            float scale;
            int sum;
            uint32_t nib[2];
            quant_group<2>(v[j], scale, sum, bad, nib);
            if (mm[j] >= 0) {
                const int mj = mm[j], g = gg[j];
                *reinterpret_cast<uint2 *>(xq + (size_t)mj * (K / 2) + (size_t)g * (kGroup / 2) + 8 * l8) =
                    make_uint2(nib[0], nib[1]);
                if (l8 == 0) {
                    sx[(size_t)mj * G + g] = scale;
                    qs[(size_t)mj * G + g] = sum;
                }
            }
        }
    }
    if (bad) flag(st, QSPEC_ERR_NONFINITE);
}

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_quant_act_int4(const uint16_t *x_bf16, int M, int K, int ldx, uint8_t *xq,
                                    float *sx, int32_t *qs, int32_t *dev_status,
                                    qspec_stream_t stream) {
    if (!x_bf16 || !xq || !sx || !qs) return QSPEC_ERR_NULL;
    if (M < 1 || K < kGroup || K % kGroup || ldx < K) return QSPEC_ERR_SHAPE;
    if ((long long)M * ((K / kGroup + 3) / 4) >= (1LL << 31)) return QSPEC_ERR_SHAPE;
    if (!aligned(x_bf16, 16) || ldx % 8 || !aligned(xq, 8) || !aligned(sx, 4) || !aligned(qs, 4))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    long long warps = (long long)M * ((K / kGroup + 3) / 4);
    long long blocks = (warps * 32 + 255) / 256;
    unsigned grid = (unsigned)std::min<long long>(blocks, (long long)sm_count() * 16);
    return launch_pdl("qspec_quant_act_int4", quant_act_kernel, dim3(grid), dim3(256), 0, as_cuda(stream),
                      x_bf16, M, K, ldx, xq, sx, qs, dev_status);
}
