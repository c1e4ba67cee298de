// Straightforward tiled ternary GEMM on CUDA cores: y[m][r] = sum_c W[r][c] * a[m][c]
// with W decoded group by group into shared memory as fp32. Correct for every
// shape and both formats; the fast decode and prefill kernels replace it on the
// shapes they cover.
#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"
#include "plane.cuh"

namespace ninfer {

constexpr int kTileRows = 64;   // weight rows per CTA
constexpr int kTileTok = 32;    // activation rows per CTA

__global__ void __launch_bounds__(256) gemm_simple_kernel(PlaneView p, uint64_t n, uint64_t k, const void *__restrict__ a,
                                                          int a_dtype, uint64_t M, void *y, int y_dtype) {
    __shared__ float Ws[kTileRows][129];
    __shared__ float As[kTileTok][129];
    const int tid = threadIdx.x;
    const uint64_t r0 = (uint64_t)blockIdx.x * kTileRows;
    const uint64_t m0 = (uint64_t)blockIdx.y * kTileTok;
    const int tx = tid & 15, ty = tid >> 4;
    float acc[2][4] = {};
    for (uint32_t gi = 0; gi < p.groups; ++gi) {
        __syncthreads();
        {   // decode 64 rows x 128 weights: thread -> row tid/4, weights 32*(tid%4) ..
            const int rr = tid >> 2, q = tid & 3;
            const uint64_t r = r0 + rr;
            if (r < n) {
                const float s = plane_scale(p, r, gi);
                for (int j = 32 * q; j < 32 * q + 32; ++j) {
                    const uint64_t c = (uint64_t)gi * 128 + j;
                    Ws[rr][j] = c < k ? (float)plane_value(p, r, gi, j) * s : 0.f;
                }
            } else {
                for (int j = 32 * q; j < 32 * q + 32; ++j) Ws[rr][j] = 0.f;
            }
        }
        for (int idx = tid; idx < kTileTok * 128; idx += 256) {
            const int mm = idx >> 7, j = idx & 127;
            const uint64_t m = m0 + mm, c = (uint64_t)gi * 128 + j;
            As[mm][j] = (m < M && c < k) ? load1(a, m * k + c, a_dtype) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < 128; ++j) {
            const float a0 = As[ty][j], a1 = As[ty + 16][j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float w = Ws[tx + 16 * q][j];
                acc[0][q] = fmaf(a0, w, acc[0][q]);
                acc[1][q] = fmaf(a1, w, acc[1][q]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t m = m0 + ty + 16 * t, r = r0 + tx + 16 * q;
            if (m < M && r < n) store1(y, m * n + r, y_dtype, acc[t][q]);
        }
}

int gemm_simple_launch(const PlaneView &p, uint64_t n, uint64_t k, const void *a, int a_dtype, uint64_t M, void *y,
                       int y_dtype, cudaStream_t stream) {
    const uint64_t gx = (n + kTileRows - 1) / kTileRows, gy = (M + kTileTok - 1) / kTileTok;
    if (gx > 0x7fffffffull || gy > 65535) return fail(NINFER_ERR_SHAPE, "matmul: problem too large for the tiled kernel");
    gemm_simple_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, stream>>>(p, n, k, a, a_dtype, M, y, y_dtype);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "matmul launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
