// Pieces shared by the fused decode kernels: the library's device error word,
// the wait bound, the once-per-kernel shared-memory attribute and tensor-map
// encoding (cached) for row-range views of a plane.
#include <cstring>
#include <unordered_map>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.h"
#include "gemv.h"

namespace ninfer {

// Error word shared by all kernels of the library (bit flags from async.cuh).
__device__ uint32_t g_device_error = 0;

int device_error_word(uint32_t **out) {
    static uint32_t *cache[64];
    static std::mutex mu;     // first calls from several host threads
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev]) {
        *out = cache[dev];
        return NINFER_OK;
    }
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "error word address: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) cache[dev] = static_cast<uint32_t *>(ptr);
    *out = static_cast<uint32_t *>(ptr);
    return NINFER_OK;
}

namespace {
std::atomic<long long> g_wait_limit{4000000000ll};
}  // namespace

long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

int set_smem_attribute(const void *kernel, int bytes) {
    struct Key {
        const void *kernel;
        int dev, bytes;
    };
    static std::mutex mu;
    static Key done[64];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev && done[i].bytes >= bytes) return NINFER_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "shared-memory attribute: %s", cudaGetErrorString(e));
    for (int i = 0; i < ndone; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev) {
            done[i].bytes = bytes;
            return NINFER_OK;
        }
    if (ndone < 64) done[ndone++] = Key{kernel, dev, bytes};
    return NINFER_OK;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_fn(EncodeTiledFn *out) {
    static EncodeTiledFn fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr)
            return fail(NINFER_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    *out = fn;
    return NINFER_OK;
}
}  // namespace

namespace {
// Encoded tensor maps, keyed by every argument of the encode. A map depends
// only on these values (an address and a shape), so a hit is always the map the
// encode would produce; calls with the same buffers skip the driver call.
struct MapKey {
    uint64_t v[14];
    bool operator==(const MapKey &o) const { return std::memcmp(v, o.v, sizeof v) == 0; }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        uint64_t h = 1469598103934665603ull;
        for (uint64_t x : k.v) h = (h ^ x) * 1099511628211ull;
        return (size_t)h;
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 4096;

bool map_lookup(const MapKey &k, CUtensorMap *out) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    auto it = g_maps.find(k);
    if (it == g_maps.end()) return false;
    *out = it->second;
    return true;
}

void map_store(const MapKey &k, const CUtensorMap &m) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
    g_maps[k] = m;
}

int encode_bytes(CUtensorMap *map, const uint8_t *addr, cuuint32_t rank, const cuuint64_t (&dims)[3],
                 const cuuint64_t (&strides)[2], uint32_t box_bytes, uint32_t box_rows, bool swizzle128) {
    const MapKey key{{1, reinterpret_cast<uint64_t>(addr), rank, dims[0], dims[1], dims[2], strides[0], strides[1],
                      box_bytes, box_rows, swizzle128 ? 1u : 0u, 0, 0, 0}};
    if (map_lookup(key, map)) return NINFER_OK;
    EncodeTiledFn fn;
    int st = encode_fn(&fn);
    if (st) return st;
    std::memset(map, 0, sizeof *map);
    const cuuint32_t box[3] = {box_bytes, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<uint8_t *>(addr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NINFER_ERR_CUDA, "tensor map encode failed (CUresult %d)", (int)r);
    map_store(key, *map);
    return NINFER_OK;
}
}  // namespace

int encode_rows(CUtensorMap *map, const uint8_t *addr, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                uint32_t box_rows, bool swizzle128) {
    const cuuint64_t dims[3] = {row_bytes, rows, 1};
    const cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
    return encode_bytes(map, addr, 2, dims, strides, box_bytes, box_rows, swizzle128);
}

int encode_row_tiles(CUtensorMap *map, const uint8_t *addr, uint64_t row_bytes, uint64_t rows, uint64_t tiles,
                     uint32_t box_bytes, uint32_t box_rows, bool swizzle128) {
    const cuuint64_t dims[3] = {row_bytes, rows, tiles};
    const cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
    return encode_bytes(map, addr, 3, dims, strides, box_bytes, box_rows, swizzle128);
}

int encode_3d_u64(CUtensorMap *map, const uint8_t *addr, const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                  const uint32_t (&box)[3]) {
    const MapKey key{{3, reinterpret_cast<uint64_t>(addr), dims[0], dims[1], dims[2], strides[0], strides[1], box[0],
                      box[1], box[2], 0, 0, 0, 0}};
    if (map_lookup(key, map)) return NINFER_OK;
    EncodeTiledFn fn;
    int st = encode_fn(&fn);
    if (st) return st;
    std::memset(map, 0, sizeof *map);
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t str[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(addr), d, str, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NINFER_ERR_CUDA, "tensor map encode failed (CUresult %d)", (int)r);
    map_store(key, *map);
    return NINFER_OK;
}

int encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *addr, uint64_t inner,
              uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    const MapKey key{{2, reinterpret_cast<uint64_t>(addr), (uint64_t)dtype, elem_bytes, inner, outer, row_stride_bytes,
                      box_inner, box_outer, swizzle128 ? 1u : 0u, 0, 0, 0, 0}};
    if (map_lookup(key, map)) return NINFER_OK;
    EncodeTiledFn fn;
    int st = encode_fn(&fn);
    if (st) return st;
    std::memset(map, 0, sizeof *map);
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void *>(addr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NINFER_ERR_CUDA, "tensor map encode failed (CUresult %d)", (int)r);
    map_store(key, *map);
    return NINFER_OK;
}

}  // namespace ninfer

extern "C" int ninfer_set_wait_limit(long long cycles) {
    if (cycles < 0) return ninfer::fail(NINFER_ERR_INVALID_ARGUMENT, "wait limit must be >= 0");
    ninfer::g_wait_limit.store(cycles == 0 ? 0 : cycles, std::memory_order_relaxed);
    return NINFER_OK;
}

extern "C" int ninfer_device_errors(uint32_t *out, int clear) {
    if (!out) return ninfer::fail(NINFER_ERR_INVALID_ARGUMENT, "device_errors: NULL output");
    cudaError_t e = cudaMemcpyFromSymbol(out, ninfer::g_device_error, sizeof(uint32_t));
    if (e != cudaSuccess) return ninfer::fail(NINFER_ERR_CUDA, "device_errors: %s", cudaGetErrorString(e));
    if (clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(ninfer::g_device_error, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return ninfer::fail(NINFER_ERR_CUDA, "device_errors: %s", cudaGetErrorString(e));
    }
    return NINFER_OK;
}
