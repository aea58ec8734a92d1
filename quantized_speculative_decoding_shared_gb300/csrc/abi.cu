// abi.cu -- version, status strings, error text, device checks.
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "qspec_host.h"

namespace qspec {

static thread_local char g_last_error[256] = "";

std::atomic<unsigned long long> &launch_count() {
    static std::atomic<unsigned long long> n{0};
    return n;
}
void count_launch() { launch_count().fetch_add(1, std::memory_order_relaxed); }

void set_last_error(const char *where, cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
             cudaGetErrorString(e));
}

static constexpr int kMaxDevices = 64;
static int g_device_ok[kMaxDevices];   // 0 unknown, 1 ok, -1 unsupported
static int g_sm_count[kMaxDevices];

int check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice", e);
        return QSPEC_ERR_LAUNCH;
    }
    if (dev < 0 || dev >= kMaxDevices) return QSPEC_ERR_UNSUPPORTED;
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = sms;
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_device_ok[dev] == 1 ? QSPEC_OK : QSPEC_ERR_UNSUPPORTED;
}

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices || g_sm_count[dev] <= 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev] = sms;
        return sms > 0 ? sms : 1;
    }
    return g_sm_count[dev];
}

// (device, kernel) pairs whose shared-memory limit is raised, with the
// bytes set; guarded by a mutex (launches may come from several threads)
struct SmemSet {
    int dev;
    const void *func;
    int bytes;
};
static constexpr int kMaxSmemSets = 256;
static SmemSet g_smem_set[kMaxSmemSets];
static int g_n_smem_set = 0;
static std::mutex g_smem_mu;

int smem_limit_once(const void *func, int bytes, bool max_carveout) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_smem_mu);
    for (int i = 0; i < g_n_smem_set; ++i)
        if (g_smem_set[i].dev == dev && g_smem_set[i].func == func && g_smem_set[i].bytes >= bytes) return QSPEC_OK;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    // optionally all of the unified L1 / shared array as shared memory, so
    // that as many CTAs as the shared memory allows can be resident
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) {
        set_last_error("cudaFuncSetAttribute", e);
        return QSPEC_ERR_LAUNCH;
    }
    for (int i = 0; i < g_n_smem_set; ++i)
        if (g_smem_set[i].dev == dev && g_smem_set[i].func == func) {
            g_smem_set[i].bytes = bytes;
            return QSPEC_OK;
        }
    if (g_n_smem_set < kMaxSmemSets) g_smem_set[g_n_smem_set++] = {dev, func, bytes};
    return QSPEC_OK;
}

int check_launch(const char *where) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_error(where, e);
        return QSPEC_ERR_LAUNCH;
    }
    return QSPEC_OK;
}

}  // namespace qspec

extern "C" {

int qspec_version(void) { return 100; }   // 0.1.0

unsigned long long qspec_kernel_launches(void) { return (unsigned long long)qspec::launch_count().load(); }

const char *qspec_status_string(int status) {
    switch (status) {
        case QSPEC_OK: return "QSPEC_OK";
        case QSPEC_ERR_NULL: return "QSPEC_ERR_NULL";
        case QSPEC_ERR_SHAPE: return "QSPEC_ERR_SHAPE";
        case QSPEC_ERR_ALIGN: return "QSPEC_ERR_ALIGN";
        case QSPEC_ERR_LAUNCH: return "QSPEC_ERR_LAUNCH";
        case QSPEC_ERR_WORKSPACE: return "QSPEC_ERR_WORKSPACE";
        case QSPEC_ERR_RANGE: return "QSPEC_ERR_RANGE";
        case QSPEC_ERR_ZERO_POINT: return "QSPEC_ERR_ZERO_POINT";
        case QSPEC_ERR_NONFINITE: return "QSPEC_ERR_NONFINITE";
        case QSPEC_ERR_TIMEOUT: return "QSPEC_ERR_TIMEOUT";
        case QSPEC_ERR_UNSUPPORTED: return "QSPEC_ERR_UNSUPPORTED";
        default: return "QSPEC_ERR_UNKNOWN";
    }
}

const char *qspec_last_cuda_error(void) { return qspec::g_last_error; }

}  // extern "C"
