// Activation preparation for the integer decode kernels: the forward signed
// block Walsh-Hadamard transform ("artifact-container.md" §8 hadamard_signs;
// TensorSharp article §4.2: per 1024-block H (D * x) / sqrt(1024)), followed by
// 16-bit fixed-point quantisation per block, laid out as dp2a operands.
//
// Output for activation row m (one region of act_prep_int16_row_bytes bytes;
// `copies` identical copies of all rows, so the many CTAs that read them spread
// over more L2 lines):
//   act[word][8] (u32): word w covers elements 16w .. 16w + 15;
//     entries 0..3 = lo_p = (x16[16w+p], x16[16w+4+p]),
//     entries 4..7 = hi_p = (x16[16w+8+p], x16[16w+12+p])   (int16 pairs)
//   gs[group] = {2^-E as float, sum of the group's x16 as int}, after act
// x16 = rint(xr * 2^E), E per block so that max |x16| < 2^14.
//
// One CTA of four warps per (block, row): thread t holds elements 8t .. 8t+7;
// index bits 0-2 are butterflied in registers, bits 3-7 across lanes and bits
// 8-9 across warps through shared memory. Computed once per call, so the decode
// kernel's CTAs only copy the finished operands.
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
namespace {

__global__ void __launch_bounds__(128) act_prep_int16_kernel(const void *__restrict__ x, int x_dtype,
                                                             const uint16_t *__restrict__ signs, uint32_t k,
                                                             uint32_t groups, uint8_t *__restrict__ out,
                                                             uint64_t row_stride_bytes, uint32_t copies,
                                                             uint64_t copy_stride_bytes) {
    __shared__ __align__(16) float xs[1024];
    __shared__ int16_t qs[1024];
    __shared__ float wmax[4];
    pdl_launch_dependents();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t b = blockIdx.x, m = blockIdx.y;
    const uint32_t c0 = b * 1024 + 8 * t;
    float d8[8];
    if (signs) load_signs8(signs, c0, d8);      // read-only parameter: before the dependency wait
    else
#pragma unroll
        for (int e = 0; e < 8; ++e) d8[e] = 1.f;
    pdl_wait();
    float v[8];
    const uint64_t xrow = (uint64_t)m * k;
    if ((b + 1) * 1024 <= k) {
        load8(x, xrow + c0, x_dtype, v);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = c0 + e < k ? load1(x, xrow + c0 + e, x_dtype) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= d8[e];
    if (signs) {
#pragma unroll
        for (int bit = 0; bit < 3; ++bit)
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (r & (1 << bit)) continue;
                const float a0 = v[r], a1 = v[r | (1 << bit)];
                v[r] = a0 + a1;
                v[r | (1 << bit)] = a0 - a1;
            }
#pragma unroll
        for (int s = 0; s < 5; ++s) {
            const bool upper = (lane >> s) & 1;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float q = __shfl_xor_sync(0xffffffffu, v[r], 1 << s);
                v[r] = upper ? (q - v[r]) : (v[r] + q);
            }
        }
    }
    *reinterpret_cast<float4 *>(&xs[8 * t]) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(&xs[8 * t + 4]) = make_float4(v[4], v[5], v[6], v[7]);
    __syncthreads();
    // element bits 8-9 (the warp index): thread (lane, warp) takes offsets
    // r = 2*warp and 2*warp+1 of lane's eight-element run in all four warps
    float u[2][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int w = 0; w < 4; ++w) u[rr][w] = xs[256 * w + 8 * lane + 2 * warp + rr];
    float mx = 0.f;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        if (signs) {
            const float a0 = u[rr][0] + u[rr][1], a1 = u[rr][0] - u[rr][1];
            const float a2 = u[rr][2] + u[rr][3], a3 = u[rr][2] - u[rr][3];
            u[rr][0] = (a0 + a2) * 0.03125f;
            u[rr][2] = (a0 - a2) * 0.03125f;
            u[rr][1] = (a1 + a3) * 0.03125f;
            u[rr][3] = (a1 - a3) * 0.03125f;
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) mx = fmaxf(mx, fabsf(u[rr][w]));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    if (lane == 0) wmax[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    int E = 0;
    if (mx > 0.f) E = 13 - ilogbf(mx);     // max |x16| < 2^14
    E = max(-100, min(100, E));
    const float up = ldexpf(1.f, E);
    // adding 1.5 * 2^23 in fp32 rounds to the nearest integer, ties to even
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int q = __float_as_int(fmaf(u[rr][w], up, 12582912.0f)) - 0x4B400000;
            qs[256 * w + 8 * lane + 2 * warp + rr] = (int16_t)q;
        }
    __syncthreads();
    // 64 words x 8 entries per block; thread t writes entries 4t .. 4t+3 (one
    // 16-byte store) into every copy of the row
    const int word = t >> 1, h = t & 1;
    const int e = 16 * word + 8 * h;
    uint4 pk;
    pk.x = (uint32_t)(uint16_t)qs[e + 0] | ((uint32_t)(uint16_t)qs[e + 4] << 16);
    pk.y = (uint32_t)(uint16_t)qs[e + 1] | ((uint32_t)(uint16_t)qs[e + 5] << 16);
    pk.z = (uint32_t)(uint16_t)qs[e + 2] | ((uint32_t)(uint16_t)qs[e + 6] << 16);
    pk.w = (uint32_t)(uint16_t)qs[e + 3] | ((uint32_t)(uint16_t)qs[e + 7] << 16);
    const bool in_row = b * 64 + word < groups * 8;      // a partial last block stops at k_pad
    for (uint32_t cp = 0; cp < copies; ++cp) {
        uint8_t *row = out + cp * copy_stride_bytes + (uint64_t)m * row_stride_bytes;
        if (in_row) reinterpret_cast<uint4 *>(row)[(b * 64 + word) * 2 + h] = pk;
    }
    // group sums: 8 groups of 128; thread t sums elements 8t .. 8t+7 (group t/16)
    int s = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) s += qs[8 * t + e];
#pragma unroll
    for (int sh = 8; sh > 0; sh >>= 1) s += __shfl_xor_sync(0xffffffffu, s, sh);
    if ((t & 15) == 0) {
        const uint32_t G = b * 8 + (t >> 4);
        if (G < groups)
            for (uint32_t cp = 0; cp < copies; ++cp) {
                uint8_t *row = out + cp * copy_stride_bytes + (uint64_t)m * row_stride_bytes;
                reinterpret_cast<float2 *>(row + (uint64_t)groups * 256)[G] = make_float2(ldexpf(1.f, -E), __int_as_float(s));
            }
    }
}

}  // namespace

uint64_t act_prep_int16_row_bytes(uint64_t k_pad) {
    const uint64_t groups = k_pad / 128;
    return ((groups * 264 + 255) / 256) * 256;
}

int act_prep_int16_launch(const void *x, int x_dtype, const uint16_t *signs, uint64_t k, uint64_t k_pad, uint64_t M,
                          uint32_t copies, uint8_t *out, cudaStream_t stream, bool pdl) {
    const uint64_t nblk = (k + 1023) / 1024;
    if (nblk > 0x7fffffffull || M > 65535) return fail(NINFER_ERR_SHAPE, "activation prep: too large");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nblk, (unsigned)M);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint64_t row_bytes = act_prep_int16_row_bytes(k_pad);
    cudaError_t e = cudaLaunchKernelEx(&cfg, act_prep_int16_kernel, x, x_dtype, signs, (uint32_t)k,
                                       (uint32_t)(k_pad / 128), out, row_bytes, copies, row_bytes * M);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "activation prep launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
