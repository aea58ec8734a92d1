// qspec_host.h -- host-side helpers of the C-ABI entry points.
#pragma once

#include <cstddef>
#include <cstdint>
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

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device and
// `slot` (each kernel variant passes its own slot < 64).  Call before a stream
// capture: the first call on a device talks to the driver.
int smem_limit_once(const void *func, int slot, int bytes);

}  // namespace qspec
