// Embedding rows: gather row ids[i] of the row-split matrix, dequantise, and
// apply the inverse signed block Hadamard transform D_b * (H e_b) / sqrt(1024)
// (TensorSharp article §4.2 inverse, §4.4 "token ID -> low-bit embedding row ->
// inverse signed Hadamard transform"). One warp per (row, 1024-block), which
// first stages that block's bytes of the row in shared memory with one vector
// load per lane.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"
#include "plane.cuh"

namespace ninfer {

// The 1024-block's payload of one row, staged per warp: PQ2_0 256 code bytes,
// or PTQ1_0 192 base bytes and 16 high bytes; then the block's 8 scales.
constexpr uint32_t kStageBytes = 256 + 16 + 16;

template <bool kPq2>
__global__ void __launch_bounds__(128) embed_kernel(PlaneView p, uint64_t n, uint64_t k, const int32_t *__restrict__ ids,
                                                    uint64_t count, const uint16_t *__restrict__ signs, void *out,
                                                    int out_dtype, int32_t *status) {
    __shared__ __align__(16) uint8_t stage_all[4][kStageBytes];
    const uint64_t nblk = k / 1024;
    const uint64_t task = (uint64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (task >= count * nblk) return;
    const int lane = threadIdx.x & 31;
    uint8_t *stage = stage_all[threadIdx.x >> 5];
    const uint64_t i = task / nblk, b = task % nblk;
    const int32_t id = ids[i];
    const bool ok = id >= 0 && (uint64_t)id < n;
    if (!ok && lane == 0 && b == 0 && status) atomicOr(status, 1);
    constexpr bool pq2 = kPq2;
    if (ok) {
        // one 8-byte load per lane: the block's codes (PQ2_0, 256 bytes) or base
        // bytes (PTQ1_0, 192), then (lanes 30, 31) its 8 high bytes' 16 and its 8 scales
        const uint32_t code_bytes = pq2 ? 256u : 192u;
        const uint8_t *row = p.base + (uint64_t)id * p.base_row + b * code_bytes;
        if (8u * lane < code_bytes) *reinterpret_cast<uint2 *>(stage + 8 * lane) = *reinterpret_cast<const uint2 *>(row + 8 * lane);
        if (lane == 30 && !pq2)
            *reinterpret_cast<uint4 *>(stage + 256) = *reinterpret_cast<const uint4 *>(p.high + (uint64_t)id * p.high_row + 16 * b);
        if (lane == 31)
            *reinterpret_cast<uint4 *>(stage + 272) = *reinterpret_cast<const uint4 *>(p.scale + (uint64_t)id * p.scale_row + 16 * b);
    }
    __syncwarp();
    // lane l holds the runs of elements 256 q + 8 l .. + 7 (q < 4): group
    // 2 q + l / 16, the same in-group positions j0 .. j0 + 7, j0 = 8 (l % 16),
    // for every q. So each of the lane's 8 positions gets its byte offset
    // (base bytes at 24 g + j / 5, high bytes at 256 + 2 g + (j - 120) / 4) and
    // its digit once; floor(byte / 3^d) = (byte * ceil(2^16 / 3^d)) >> 16 and
    // q % 3 = q - 3 ((q * 21846) >> 16) are exact for every byte value, d <= 4.
    float v[32];
    const int j0 = 8 * (lane & 15);
    int off[8];
    uint32_t mul[8];
    bool high[8];
#pragma unroll
    for (int e = 0; e < 8 && !pq2; ++e) {
        const int j = j0 + e;
        high[e] = j >= 120;
        const int d = high[e] ? (j - 120) & 3 : j % 5;
        off[e] = high[e] ? 256 + ((j - 120) >> 2) : j / 5;
        mul[e] = d == 0 ? 65536u : d == 1 ? 21846u : d == 2 ? 7282u : d == 3 ? 2428u : 810u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int g = 2 * q + (lane >> 4);
        const float s = __half2float(*reinterpret_cast<const __half *>(stage + 272 + 2 * g));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            int val;
            if (pq2) {
                const int c = 256 * q + 8 * lane + e;
                val = (int)((stage[c >> 2] >> (2 * (c & 3))) & 3u) - 1;
            } else {
                const uint32_t byte = stage[off[e] + (high[e] ? 2 * g : 24 * g)];
                const uint32_t t = (byte * mul[e]) >> 16;
                val = (int)(t - 3 * ((t * 21846u) >> 16)) - 1;
            }
            v[8 * q + e] = ok ? (float)val * s : 0.f;
        }
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
        if (fmt == NINFER_PQ2_0_G128)
            embed_kernel<true><<<(unsigned)grid, 128, 0, s>>>(p, n, k, ids, count, signs_bf16, out, out_dtype, status_dev);
        else
            embed_kernel<false><<<(unsigned)grid, 128, 0, s>>>(p, n, k, ids, count, signs_bf16, out, out_dtype, status_dev);
    } else {
        const uint64_t total = count * k, grid = (total + 255) / 256;
        if (grid > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "embed: too many rows");
        embed_plain_kernel<<<(unsigned)grid, 256, 0, s>>>(p, n, k, ids, count, out, out_dtype, status_dev);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "embed launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}
