// Device helpers: element loads/stores by dtype and the 1024-point
// Walsh-Hadamard butterfly held by one warp.
//
// Hadamard convention ("artifact-container.md" §8 hadamard_signs; TensorSharp
// article §4.2): H is the unnormalised Sylvester matrix in natural order,
// H[i][j] = (-1)^popcount(i & j), so the transform is a product of independent
// 2-point butterflies (a, b) -> (a + b, a - b), one per index bit.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ninfer_ternary.h"

namespace ninfer {

// Warp-owned 1024-element block: lane l holds v[8*i + e] = element
// 256*i + 8*l + e (i < 4, e < 8). Index bits 0-2 and 8-9 live in the lane's
// registers, bits 3-7 in the lane id.

__device__ __forceinline__ void wht1024_warp(float (&v)[32], int lane) {
#pragma unroll
    for (int b = 0; b < 5; ++b) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j & (1 << b)) continue;
            const float a = v[j], c = v[j | (1 << b)];
            v[j] = a + c;
            v[j | (1 << b)] = a - c;
        }
    }
    // lane bits: the lane whose bit s is set keeps partner - own, the other own +
    // partner; fmaf(+-1, own, partner) rounds once, exactly as that add does.
    // One rolled loop keeps the code (fetched once per launch) short.
#pragma unroll 1
    for (int s = 0; s < 5; ++s) {
        const float sg = ((lane >> s) & 1) ? -1.f : 1.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float p = __shfl_xor_sync(0xffffffffu, v[j], 1 << s);
            v[j] = fmaf(sg, v[j], p);
        }
    }
}

// 8 consecutive elements (16-byte aligned) -> fp32.
__device__ __forceinline__ void load8(const void *base, uint64_t idx, int dtype, float (&o)[8]) {
    if (dtype == NINFER_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx);
        float4 a = __ldg(p), b = __ldg(p + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + idx));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (dtype == NINFER_BF16) {
                o[2 * q] = __uint_as_float(w[q] << 16);
                o[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
            } else {
                __half2 h = *reinterpret_cast<const __half2 *>(&w[q]);
                float2 f = __half22float2(h);
                o[2 * q] = f.x;
                o[2 * q + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ void store8(void *base, uint64_t idx, int dtype, const float (&o)[8]) {
    if (dtype == NINFER_F32) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(base) + idx);
        p[0] = make_float4(o[0], o[1], o[2], o[3]);
        p[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (dtype == NINFER_BF16) {
                __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * q], o[2 * q + 1]);
                w[q] = *reinterpret_cast<uint32_t *>(&h);
            } else {
                __half2 h = __floats2half2_rn(o[2 * q], o[2 * q + 1]);
                w[q] = *reinterpret_cast<uint32_t *>(&h);
            }
        }
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ float load1(const void *base, uint64_t idx, int dtype) {
    if (dtype == NINFER_F32) return static_cast<const float *>(base)[idx];
    const uint16_t h = static_cast<const uint16_t *>(base)[idx];
    if (dtype == NINFER_BF16) return __uint_as_float((uint32_t)h << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void store1(void *base, uint64_t idx, int dtype, float v) {
    if (dtype == NINFER_F32) static_cast<float *>(base)[idx] = v;
    else if (dtype == NINFER_BF16) static_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(v);
    else static_cast<__half *>(base)[idx] = __float2half_rn(v);
}

// Sign vector (bfloat16 +-1): 8 consecutive entries as fp32.
__device__ __forceinline__ void load_signs8(const uint16_t *s, uint64_t idx, float (&o)[8]) { load8(s, idx, NINFER_BF16, o); }

inline size_t dtype_size(int dt) { return dt == NINFER_F32 ? 4 : 2; }
inline bool dtype_valid(int dt) { return dt == NINFER_F32 || dt == NINFER_BF16 || dt == NINFER_F16; }

}  // namespace ninfer
