// kv.cu -- a7: KV-cache overwrite at accepted positions.
//
// QSPEC summary page, "QSPEC structure": for accepted tokens the KV-cache
// entries written by the W4A4 draft pass are replaced with the W4A16 verify
// pass's, so later decoding reads high-quality context from the one shared
// cache (no second cache is kept).  Positions base_pos[b] .. base_pos[b] +
// n_acc[b] are rewritten: the last confirmed token (whose K/V the first draft
// step wrote) and the accepted drafts.
//
// Pure copy, HBM-bound: 16-byte loads and stores; consecutive threads walk one
// D-row, then the heads of a position (contiguous in the verify-pass layout).
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

__global__ void __launch_bounds__(256) kv_overwrite_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                                          const uint4 *__restrict__ kn,
                                                          const uint4 *__restrict__ vn,
                                                          const int32_t *__restrict__ base_pos,
                                                          const int32_t *__restrict__ n_acc, int L, int B,
                                                          int H, int T, int D, int gamma, int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    const int D8 = D / 8;
    const long long total = (long long)L * B * (gamma + 1) * H * D8;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long t = i;
        const int c = (int)(t % D8); t /= D8;
        const int h = (int)(t % H); t /= H;
        const int r = (int)(t % (gamma + 1)); t /= (gamma + 1);
        const int b = (int)(t % B);
        const int l = (int)(t / B);
        const int p0 = base_pos[b], a = n_acc[b];
        if (p0 < 0 || a < 0 || a > gamma || p0 + a >= T) {
            if (l == 0 && r == 0 && h == 0 && c == 0) flag(st, QSPEC_ERR_RANGE);
            continue;
        }
        if (r > a) continue;
        const size_t src = ((((size_t)l * B + b) * (gamma + 1) + r) * H + h) * D8 + c;
        const size_t dst = ((((size_t)l * B + b) * H + h) * T + (size_t)(p0 + r)) * D8 + c;
        kc[dst] = __ldcs(kn + src);
        vc[dst] = __ldcs(vn + src);
    }
}

}  // namespace qspec

using namespace qspec;

extern "C" int qspec_kv_overwrite(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                                  const uint16_t *v_new, const int32_t *base_pos, const int32_t *n_acc,
                                  int L, int B, int H, int T, int D, int gamma, int32_t *dev_status,
                                  qspec_stream_t stream) {
    if (!k_cache || !v_cache || !k_new || !v_new || !base_pos || !n_acc) return QSPEC_ERR_NULL;
    if (L < 1 || B < 1 || H < 1 || T < 1 || D < 8 || D % 8 || gamma < 0 || gamma > QSPEC_MAX_GAMMA)
        return QSPEC_ERR_SHAPE;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(base_pos, 4) || !aligned(n_acc, 4))
        return QSPEC_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    long long total = (long long)L * B * (gamma + 1) * H * (D / 8);
    unsigned grid = (unsigned)std::min<long long>((total + 255) / 256, (long long)sm_count() * 16);
    return launch_pdl("qspec_kv_overwrite", kv_overwrite_kernel, dim3(grid), dim3(256), 0, as_cuda(stream),
                      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
                      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), base_pos,
                      n_acc, L, B, H, T, D, gamma, dev_status);
}
