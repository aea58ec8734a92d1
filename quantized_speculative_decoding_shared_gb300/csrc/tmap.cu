// tmap.cu -- host side of the TMA weight loads: 2-D tensor maps over packed
// INT4 weight matrices ([N rows][K / 2 bytes]), cached per (address, N, K).
#include <cstring>
#include <mutex>

#include "qspec_host.h"

namespace qspec {

namespace {

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

struct Entry {
    const void *ptr;
    int n, k, box_rows, dev;
    CUtensorMap map;
};
constexpr int kEntries = 256;
Entry g_cache[kEntries];
int g_next = 0;
std::mutex g_mu;

}  // namespace

int weight_tmap(CUtensorMap *out, const uint8_t *packed, int N, int K, int box_rows) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < kEntries; ++i) {
        const Entry &e = g_cache[i];
        if (e.ptr == packed && e.n == N && e.k == K && e.box_rows == box_rows && e.dev == dev) {
            *out = e.map;
            return QSPEC_OK;
        }
    }
    EncodeTiled fn = encoder();
    if (!fn) return QSPEC_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(packed), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return QSPEC_ERR_UNSUPPORTED;
    Entry &e = g_cache[g_next];
    g_next = (g_next + 1) % kEntries;
    e.ptr = packed;
    e.n = N;
    e.k = K;
    e.box_rows = box_rows;
    e.dev = dev;
    e.map = map;
    *out = map;
    return QSPEC_OK;
}

// 2-D TMA map over a row-major byte matrix [rows][cols] with rows `pitch`
// bytes apart: boxes of 128 bytes x box_rows rows, 128-byte swizzle, rows
// and columns past the matrix read as zeros.  Not cached (for per-call
// operands); QSPEC_ERR_UNSUPPORTED if the driver refuses the map.
int byte_tmap_sw128(CUtensorMap *out, const void *base, int rows, int cols, size_t pitch, int box_rows) {
    EncodeTiled fn = encoder();
    if (!fn) return QSPEC_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    std::memset(out, 0, sizeof(*out));
    CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QSPEC_OK : QSPEC_ERR_UNSUPPORTED;
}

}  // namespace qspec
