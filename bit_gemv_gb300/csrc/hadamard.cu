// Signed block Walsh-Hadamard transform, forward and inverse.
//
// Forward ("artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2):
//   per 1024-block b of each row: y_b = H (D_b * x_b) / sqrt(1024)
// Inverse (TensorSharp article §4.2, applied to embedding rows):
//   y_b = D_b * (H x_b) / sqrt(1024)
// One warp per (row, block); memory-bound: each block reads 1024 inputs and
// 1024 signs and writes 1024 outputs with 16-byte vector accesses.
#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"

namespace ninfer {

template <bool kInverse>
__global__ void __launch_bounds__(128) hadamard_kernel(const void *__restrict__ x, int x_dtype, void *y, int y_dtype,
                                                       const uint16_t *__restrict__ signs, uint64_t M, uint64_t K) {
    const uint64_t nblk = K / 1024;
    const uint64_t task = (uint64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (task >= M * nblk) return;
    const int lane = threadIdx.x & 31;
    const uint64_t m = task / nblk, b = task % nblk;
    const uint64_t row = m * K, col0 = b * 1024;
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float t[8], d[8];
        const uint64_t c = col0 + 256 * i + 8 * lane;
        load8(x, row + c, x_dtype, t);
        if (!kInverse) {
            load_signs8(signs, c, d);
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] *= d[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * i + e] = t[e];
    }
    wht1024_warp(v, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float t[8], d[8];
        const uint64_t c = col0 + 256 * i + 8 * lane;
        if (kInverse) load_signs8(signs, c, d);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = v[8 * i + e] * 0.03125f * (kInverse ? d[e] : 1.0f);
        store8(y, row + c, y_dtype, t);
    }
}

static int hadamard_launch(bool inverse, const void *x, int x_dtype, void *y, int y_dtype, const uint16_t *signs,
                           uint64_t M, uint64_t K, cudaStream_t stream) {
    if (!x || !y || !signs) return fail(NINFER_ERR_INVALID_ARGUMENT, "hadamard: NULL pointer");
    if (!dtype_valid(x_dtype) || !dtype_valid(y_dtype)) return fail(NINFER_ERR_INVALID_ARGUMENT, "hadamard: bad dtype");
    if (M == 0 || K == 0) return fail(NINFER_ERR_SHAPE, "hadamard: M and K must be positive");
    if (K % 1024) return fail(NINFER_ERR_SHAPE, "hadamard: K=%llu is not a multiple of the 1024-element block",
                              (unsigned long long)K);
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(signs, 16))
        return fail(NINFER_ERR_ALIGNMENT, "hadamard: x, y and signs must be 16-byte aligned");
    if (x == y && x_dtype != y_dtype) return fail(NINFER_ERR_INVALID_ARGUMENT, "hadamard: in-place needs equal dtypes");
    const uint64_t tasks = M * (K / 1024);
    const uint64_t grid = (tasks + 3) / 4;
    if (grid > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "hadamard: too many blocks");
    if (inverse)
        hadamard_kernel<true><<<(unsigned)grid, 128, 0, stream>>>(x, x_dtype, y, y_dtype, signs, M, K);
    else
        hadamard_kernel<false><<<(unsigned)grid, 128, 0, stream>>>(x, x_dtype, y, y_dtype, signs, M, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "hadamard launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer

extern "C" int ninfer_hadamard_fwd(const void *x, int x_dtype, void *y, int y_dtype, const uint16_t *signs_bf16,
                                   uint64_t M, uint64_t K, ninfer_stream stream) {
    return ninfer::hadamard_launch(false, x, x_dtype, y, y_dtype, signs_bf16, M, K, (cudaStream_t)stream);
}

extern "C" int ninfer_hadamard_inv(const void *x, int x_dtype, void *y, int y_dtype, const uint16_t *signs_bf16,
                                   uint64_t M, uint64_t K, ninfer_stream stream) {
    return ninfer::hadamard_launch(true, x, x_dtype, y, y_dtype, signs_bf16, M, K, (cudaStream_t)stream);
}
