// bounded.cu -- qspec_debug_linear_bounded: one tensor-core linear kernel
// with a chosen bound on its barrier waits and, optionally, a wait that is
// made to run out, so that the timeout exit (status, drain, tensor memory
// freed, context still usable) can be tested without any fault.
#include "qspec_device.cuh"
#include "qspec_host.h"

using namespace qspec;

extern "C" int qspec_debug_linear_bounded(int kernel, const uint16_t *x_bf16, const uint8_t *xq, const float *sx,
                                          const int32_t *qs, const uint8_t *packed, const uint32_t *sz, int M,
                                          int N, int K, uint16_t *y_bf16, int ldy, uint32_t wait_limit, int stall,
                                          int32_t *dev_status, qspec_stream_t stream) {
    if (!packed || !sz || !y_bf16) return QSPEC_ERR_NULL;
    if (M < 1 || N < 1 || K < QSPEC_GROUP || K % QSPEC_GROUP || ldy < N || wait_limit < 1) return QSPEC_ERR_SHAPE;
    if (!aligned(packed, 16) || !aligned(sz, 4) || !aligned(y_bf16, 2)) return QSPEC_ERR_ALIGN;
    const bool w4a16 = kernel == QSPEC_KERNEL_W4A16_TC;
    if (w4a16) {
        if (!x_bf16) return QSPEC_ERR_NULL;
        if (!aligned(x_bf16, 16)) return QSPEC_ERR_ALIGN;
    } else {
        if (!xq || !sx || !qs) return QSPEC_ERR_NULL;
        if (!aligned(xq, 16) || !aligned(sx, 4) || !aligned(qs, 4)) return QSPEC_ERR_ALIGN;
    }
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = as_cuda(stream);
    switch (kernel) {
        case QSPEC_KERNEL_W4A16_TC:
            return launch_w4a16_tc(x_bf16, K, packed, sz, M, N, K, y_bf16, ldy, dev_status, st, wait_limit, stall,
                                   KvOut{nullptr, nullptr, nullptr, nullptr, 0, 1, 1, 1, 0, nullptr});
        case QSPEC_KERNEL_W4A4_GEMV_TC:
            return launch_w4a4_gemv_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, nullptr, dev_status, st,
                                       wait_limit, stall);
        case QSPEC_KERNEL_W4A4_TC:
            return launch_w4a4_tc(xq, sx, qs, packed, sz, M, N, K, y_bf16, ldy, nullptr, dev_status, st, wait_limit,
                                  stall);
        default:
            return QSPEC_ERR_SHAPE;
    }
}
