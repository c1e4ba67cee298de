// Embedding rows: gather row ids[i] of the row-split matrix, dequantise, and
// apply the inverse signed block Hadamard transform D_b * (H e_b) / sqrt(1024)
// (TensorSharp article §4.2 inverse, §4.4 "token ID -> low-bit embedding row ->
// inverse signed Hadamard transform"). One warp per (row, 1024-block).
#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"
#include "plane.cuh"

namespace ninfer {

__global__ void __launch_bounds__(128) embed_kernel(PlaneView p, uint64_t n, uint64_t k, const int32_t *__restrict__ ids,
                                                    uint64_t count, const uint16_t *__restrict__ signs, void *out,
                                                    int out_dtype, int32_t *status) {
    const uint64_t nblk = k / 1024;
    const uint64_t task = (uint64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (task >= count * nblk) return;
    const int lane = threadIdx.x & 31;
    const uint64_t i = task / nblk, b = task % nblk;
    const int32_t id = ids[i];
    const bool ok = id >= 0 && (uint64_t)id < n;
    if (!ok && lane == 0 && b == 0 && status) atomicOr(status, 1);
    float v[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const uint64_t c = b * 1024 + wht_index(lane, r);
        const uint32_t gi = (uint32_t)(c >> 7);
        v[r] = ok ? (float)plane_value(p, (uint64_t)id, gi, (int)(c & 127)) * plane_scale(p, (uint64_t)id, gi) : 0.f;
    }
    wht1024_warp(v, lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float t[8], d[8];
        const uint64_t c = b * 1024 + 256 * q + 8 * lane;
        load_signs8(signs, c, d);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = ok ? v[8 * q + e] * 0.03125f * d[e] : 0.f;
        store8(out, i * k + c, out_dtype, t);
    }
}

// Dequantise only (no transform): one thread per output element.
__global__ void embed_plain_kernel(PlaneView p, uint64_t n, uint64_t k, const int32_t *__restrict__ ids, uint64_t count,
                                   void *out, int out_dtype, int32_t *status) {
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= count * k) return;
    const uint64_t i = t / k, c = t % k;
    const int32_t id = ids[i];
    const bool ok = id >= 0 && (uint64_t)id < n;
    if (!ok && c == 0 && status) atomicOr(status, 1);
    const uint32_t gi = (uint32_t)(c >> 7);
    const float v = ok ? (float)plane_value(p, (uint64_t)id, gi, (int)(c & 127)) * plane_scale(p, (uint64_t)id, gi) : 0.f;
    store1(out, t, out_dtype, v);
}

}  // namespace ninfer

using namespace ninfer;

extern "C" int ninfer_ternary_embed(int fmt, const uint8_t *payload, uint64_t payload_bytes, uint64_t n, uint64_t k,
                                    const int32_t *ids, uint64_t count, const uint16_t *signs_bf16, void *out,
                                    int out_dtype, int32_t *status_dev, ninfer_stream stream) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!payload || !ids || !out) return fail(NINFER_ERR_INVALID_ARGUMENT, "embed: NULL pointer");
    if (count == 0) return fail(NINFER_ERR_SHAPE, "embed: count must be positive");
    if (out_dtype != NINFER_F32 && out_dtype != NINFER_BF16)
        return fail(NINFER_ERR_INVALID_ARGUMENT, "embed: out dtype must be f32 or bf16");
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    if (!aligned(payload, 256)) return fail(NINFER_ERR_ALIGNMENT, "embed: payload must be 256-byte aligned");
    if (!aligned(out, 16) || !aligned(ids, 4) || (signs_bf16 && !aligned(signs_bf16, 16)))
        return fail(NINFER_ERR_ALIGNMENT, "embed: out and signs must be 16-byte aligned");
    const PlaneView p = make_view(payload, g, fmt);
    cudaStream_t s = (cudaStream_t)stream;
    if (signs_bf16) {
        if (k % 1024) return fail(NINFER_ERR_SHAPE, "embed: k=%llu is not a multiple of 1024", (unsigned long long)k);
        const uint64_t tasks = count * (k / 1024), grid = (tasks + 3) / 4;
        if (grid > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "embed: too many rows");
        embed_kernel<<<(unsigned)grid, 128, 0, s>>>(p, n, k, ids, count, signs_bf16, out, out_dtype, status_dev);
    } else {
        const uint64_t total = count * k, grid = (total + 255) / 256;
        if (grid > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "embed: too many rows");
        embed_plain_kernel<<<(unsigned)grid, 256, 0, s>>>(p, n, k, ids, count, out, out_dtype, status_dev);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "embed launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}
