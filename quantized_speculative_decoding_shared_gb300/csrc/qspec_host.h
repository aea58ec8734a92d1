// qspec_host.h -- host-side helpers of the C-ABI entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "qspec.h"

namespace qspec {

// Records a CUDA error text for qspec_last_cuda_error() (per calling thread).
void set_last_error(const char *where, cudaError_t e);

// QSPEC_OK when the current device is an sm_103 part (checked once per device),
// else QSPEC_ERR_UNSUPPORTED or QSPEC_ERR_LAUNCH.
int check_device();

// QSPEC_OK, or QSPEC_ERR_LAUNCH if the launch just made failed.
int check_launch(const char *where);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t as_cuda(qspec_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` (with
// max_carveout, also prefer the largest shared-memory carveout), once per
// device and kernel.  Call before a stream capture: the first call for a
// kernel on a device talks to the driver.
int smem_limit_once(const void *func, int bytes, bool max_carveout = false);

// One-token W4A4 on the byte dot-product unit (w4a4_dp4a.cu): xq, sx, qs as
// input, or x (bf16) quantised in the kernel with xq_out, sx_out, qs_out
// stored; QSPEC_ERR_SHAPE before any launch when K does not suit it.
int launch_w4a4_dp4a(const uint8_t *xq, const float *sx, const int32_t *qs, const uint16_t *x, uint8_t *xq_out,
                     float *sx_out, int32_t *qs_out, const uint8_t *packed, const uint32_t *sz, int N, int K,
                     uint16_t *y, int32_t *dbg_I, int32_t *dev_status, cudaStream_t stream);

// The tensor-core kernels below bound every barrier wait by wait_limit polls
// (kWaitLimit in the regular calls); stall != 0 (tests only) makes the MMA
// issuer first wait on a barrier nothing arrives at, so that the wait runs
// out and the kernel takes its timeout exit.

// Large-M W4A16 on the tensor cores (w4a16_tc.cu); kv: the optional cache
// output of the epilogue (KvOut in qspec_device.cuh).
struct KvOut;
int launch_w4a16_tc(const uint16_t *x, int ldx, const uint8_t *packed, const uint32_t *sz, int M, int N, int K,
                    uint16_t *y, int ldy, int32_t *st, cudaStream_t stream, uint32_t wait_limit, int stall,
                    const KvOut &kv);

// Larger-M W4A4 on the tensor cores (w4a4_tc.cu).
int launch_w4a4_tc(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                   const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st,
                   cudaStream_t stream, uint32_t wait_limit, int stall);
int launch_w4a4_tc_wide(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                   const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I, int32_t *st,
                   cudaStream_t stream, uint32_t wait_limit, int stall);

// Decode-sized W4A4 (3 <= M <= 16) on the tensor cores with the weights
// staged in TMEM (w4a4_gemv_tc.cu); QSPEC_ERR_SHAPE before any launch when
// the shape does not suit it.
int launch_w4a4_gemv_tc(const uint8_t *xq, const float *sx, const int32_t *qs, const uint8_t *packed,
                        const uint32_t *sz, int M, int N, int K, uint16_t *y, int ldy, int32_t *dbg_I,
                        int32_t *dev_status, cudaStream_t stream, uint32_t wait_limit, int stall);

// 2-D TMA map over a packed weight matrix [N][K / 2] bytes: boxes of 128
// bytes x box_rows rows, 128-byte swizzle, rows past N read as zeros.
int weight_tmap(CUtensorMap *out, const uint8_t *packed, int N, int K, int box_rows);

// 2-D TMA map over a row-major byte matrix [rows][cols], rows `pitch` bytes
// apart: boxes of 128 bytes x box_rows rows, 128-byte swizzle, reads past
// the matrix give zeros (not cached).
int byte_tmap_sw128(CUtensorMap *out, const void *base, int rows, int cols, size_t pitch, int box_rows);

// Polls of a bounded barrier wait in the tensor-core kernels (each poll
// suspends for a hardware-chosen time); a wait that runs out sets
// QSPEC_ERR_TIMEOUT.
constexpr uint32_t kWaitLimit = 1u << 22;


// One more kernel launch issued (the count qspec_kernel_launches reports).
void count_launch();

// Launch `kernel` on `st` with programmatic stream serialisation allowed (the
// kernel must follow the pdl_wait() rule in qspec_device.cuh).
template <typename... KArgs, typename... Args>
int launch_pdl(const char *where, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
               cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) {
        set_last_error(where, e);
        return QSPEC_ERR_LAUNCH;
    }
    count_launch();
    return QSPEC_OK;
}

// The same with thread-block clusters of `cluster_x` CTAs along x (grid.x a
// multiple of it).
template <typename... KArgs, typename... Args>
int launch_pdl_cluster(const char *where, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) {
        set_last_error(where, e);
        return QSPEC_ERR_LAUNCH;
    }
    count_launch();
    return QSPEC_OK;
}

}  // namespace qspec
