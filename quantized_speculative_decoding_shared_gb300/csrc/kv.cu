// kv.cu -- a7: KV-cache overwrite at accepted positions.
//
// QSPEC summary page, "QSPEC structure": for accepted tokens the KV-cache
// entries written by the W4A4 draft pass are replaced with the W4A16 verify
// pass's, so later decoding reads high-quality context from the one shared
// cache (no second cache is kept).  Positions base_pos[b] .. base_pos[b] +
// n_acc[b] are rewritten: the last confirmed token (whose K/V the first draft
// step wrote) and the accepted drafts.
//
// Pure copy, HBM-bound: 16-byte loads and stores; one CTA per (layer,
// sequence, verify row), whose threads walk the H x D row (contiguous in the
// verify-pass layout); rows past the accepted count return at once.
#include <algorithm>

#include "qspec_device.cuh"
#include "qspec_host.h"

namespace qspec {

// one CTA per (layer, sequence, verify row); its threads copy the H x D row
// in 16-byte pieces (no per-element index arithmetic beyond one division)
constexpr int kKvThreads = 128;

__global__ void __launch_bounds__(kKvThreads) kv_overwrite_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                                                 const uint4 *__restrict__ kn,
                                                                 const uint4 *__restrict__ vn,
                                                                 const int32_t *__restrict__ base_pos,
                                                                 const int32_t *__restrict__ n_acc, int L, int B,
                                                                 int H, int T, int D, int gamma, int32_t *st) {
    pdl_launch_dependents();
    pdl_wait();
    const int D8 = D / 8, R = gamma + 1;
    const int blk = blockIdx.x;                       // = (l * B + b) * R + r
    const int r = blk % R, lb = blk / R, b = lb % B, l = lb / B;
    const int p0 = base_pos[b], a = n_acc[b];
    if (p0 < 0 || a < 0 || a > gamma || p0 + a >= T) {
        if (l == 0 && r == 0 && threadIdx.x == 0) flag(st, QSPEC_ERR_RANGE);
        return;
    }
    if (r > a) return;
    const uint4 *ks = kn + (size_t)blk * H * D8, *vs = vn + (size_t)blk * H * D8;
    const size_t head0 = ((size_t)l * B + b) * H;       // (l, b, h = 0) row of the cache
    for (int e = threadIdx.x; e < H * D8; e += kKvThreads) {
        const int h = e / D8, c = e - h * D8;
        const size_t dst = ((head0 + h) * T + (size_t)(p0 + r)) * D8 + c;
        kc[dst] = __ldcs(ks + e);
        vc[dst] = __ldcs(vs + e);
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
    const long long blocks = (long long)L * B * (gamma + 1);
    if (blocks >= (1LL << 31) || (long long)H * (D / 8) >= (1LL << 31)) return QSPEC_ERR_SHAPE;
    return launch_pdl("qspec_kv_overwrite", kv_overwrite_kernel, dim3((unsigned)blocks), dim3(kKvThreads), 0,
                      as_cuda(stream),
                      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
                      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), base_pos,
                      n_acc, L, B, H, T, D, gamma, dev_status);
}
