// ninfer_ternary_matmul_noalloc: the projection for callers that cannot
// allocate device memory themselves.
//
// Some callers have no way to call cudaMalloc (or any allocator) around a
// projection: code running under an allocator-less runtime, plugins handed
// only pre-placed input/output buffers by their host, or a process whose
// memory budget is fixed before it starts. ninfer_ternary_matmul needs a
// caller-provided workspace on the paths that stage rotated activations; this
// entry point supplies that workspace from a fixed array in the library's own
// device memory instead. The array is a file-scope __device__ object, so every
// GPU that loads the library holds it until the process exits.
//
// Host code must not hand the array's name to a kernel: on the host that name
// is only a stand-in symbol. Its device address is obtained once per device
// with cudaGetSymbolAddress (on the first call made with that device current)
// and cached for the life of the process, so calls must not cross a
// cudaDeviceReset (or any other teardown of the device's primary context): the
// library is loaded again into the new context and the cached address would
// be stale. The first call on a device should also come before any stream
// capture, since it does this set-up.
#include <mutex>

#include <cuda_runtime.h>

#include "common.h"

namespace ninfer {
namespace {

constexpr uint64_t kNoAllocScratchBytes = NINFER_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set-up once per
// device, with that device current).
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(NINFER_ERR_CUDA, "noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(NINFER_ERR_CUDA, "noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                        cudaGetErrorString(e));
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return NINFER_OK;
}

}  // namespace
}  // namespace ninfer

extern "C" int ninfer_ternary_matmul_noalloc(int fmt, const uint8_t *payload, uint64_t payload_bytes, uint64_t n,
                                             uint64_t k, const void *x, int x_dtype, const uint16_t *signs_bf16,
                                             void *y, int y_dtype, uint64_t M, ninfer_stream stream) {
    using namespace ninfer;
    if (M == 0) return fail(NINFER_ERR_SHAPE, "noalloc: M must be positive");
    uint64_t need = 0;
    int st = ninfer_ternary_matmul_workspace(fmt, n, k, M, signs_bf16 != nullptr, &need);
    if (st) return st;
    if (need > kNoAllocScratchBytes)
        return fail(NINFER_ERR_SIZE_MISMATCH,
                    "noalloc: this problem needs %llu bytes of scratch; the built-in array holds %llu "
                    "(use ninfer_ternary_matmul with a caller workspace)",
                    (unsigned long long)need, (unsigned long long)kNoAllocScratchBytes);
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st) return st;
    // Nothing is cleared between calls: every path writes each workspace byte
    // it later reads, within the same call, before reading it. The users are
    // the rotated or packed activations (all paths that stage them), the
    // binary16 MMA fragments (PQ2_0, 2 <= M <= 8), the per-block fp32 partial
    // sums (PTQ1_0, 2 <= M <= 8; padded rows that no block writes are never
    // read back) and the PTQ1_0 planes rewritten as PQ2_0 planes (prefill).
    return ninfer_ternary_matmul(fmt, payload, payload_bytes, n, k, x, x_dtype, signs_bf16, y, y_dtype, M, scratch,
                                 kNoAllocScratchBytes, stream);
}
