// Activation helpers shared by the decode kernels: the dp2a wrappers of the
// M = 1 integer kernels, and for the M <= 8 tensor-core kernels the loads of a
// 1024-block of x and its signs and the forward signed block Walsh-Hadamard
// transform ("artifact-container.md" §8 hadamard_signs; TensorSharp article
// §4.2: per 1024-block H (D * x) / 32).
//
// rotate16: two warps (64 threads) per 1024-block, 16 elements per thread, in
// three register passes over index bits 0-3, 4-7 and 8-9 with transposes
// through a padded float tile between them (element e at e + e/16,
// conflict-free for the first two layouts). Each kernel then converts the
// rotated values into its own operand layout.
#pragma once

#include <cstdint>

#include "async.cuh"
#include "device.cuh"

namespace ninfer {

constexpr uint32_t kRotScratch = (1024 + 64) * 4 + 16;     // bytes per rotating warp pair

struct XSource {
    const void *x;
    const uint16_t *signs;     // bf16 +-1 per element, or null (no rotation)
    uint32_t k;
    int x_dtype;
};

__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int pad16(int e) { return e + (e >> 4); }

// x of block b: thread t (0..63) gets elements 16t .. 16t + 15 (zero past k).
__device__ __forceinline__ void load_run16(const XSource &xs, uint32_t b, int t, float (&v)[16]) {
    const uint64_t e0 = (uint64_t)b * 1024 + 16 * t;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float u[8];
        const uint64_t idx = e0 + 8 * i;
        if (idx + 8 <= xs.k) {
            load8(xs.x, idx, xs.x_dtype, u);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = idx + e < xs.k ? load1(xs.x, idx + e, xs.x_dtype) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * i + e] = u[e];
    }
}

__device__ __forceinline__ void load_signs16(const XSource &xs, uint32_t b, int t, float (&d)[16]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float u[8];
        load_signs8(xs.signs, (uint64_t)b * 1024 + 16 * t + 8 * i, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) d[8 * i + e] = u[e];
    }
}

// Butterflies over register index bits kLo .. kLo + kBits - 1 of 16 values.
template <int kLo, int kBits>
__device__ __forceinline__ void butterfly16(float (&v)[16]) {
#pragma unroll
    for (int bit = kLo; bit < kLo + kBits; ++bit)
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if (r & (1 << bit)) continue;
            const float a0 = v[r], a1 = v[r | (1 << bit)];
            v[r] = a0 + a1;
            v[r | (1 << bit)] = a0 - a1;
        }
}

// Rotates block b (x in v, signs in d) in place: on return v[r] holds xr of
// element 256 (r / 4) + 4t + r % 4, and the return value is the block's
// largest |xr|. The tile's first 1088 floats are free again; the two after
// them hold the warps' maxima until the pair's next barrier. t = thread of the
// pair (0..63), bar = the pair's named barrier.
__device__ __forceinline__ float rotate16(bool rotate, int t, float (&v)[16], const float (&d)[16], float *tile,
                                          uint32_t bar) {
    const int lane = t & 31;
    float *pmax = tile + 1024 + 64;
    if (rotate) {
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] *= d[r];
        butterfly16<0, 4>(v);                                    // bits 0-3: elements 16t + r
#pragma unroll
        for (int r = 0; r < 16; ++r) tile[17 * t + r] = v[r];      // pad16(16t + r)
        named_barrier(bar, 64);
        // bits 4-7: thread t = (hi2, lo4) takes elements 256 hi2 + 16 r + lo4
        const int hi2 = t >> 4, lo4 = t & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = tile[272 * hi2 + 17 * r + lo4];
        butterfly16<0, 4>(v);
#pragma unroll
        for (int r = 0; r < 16; ++r) tile[272 * hi2 + 17 * r + lo4] = v[r];
        named_barrier(bar, 64);
        // bits 8-9: thread t takes elements 256 a + 4t + c (a = r / 4, c = r % 4)
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = tile[pad16(256 * (r >> 2) + 4 * t + (r & 3))];
        butterfly16<2, 2>(v);                                    // register bits 2-3 = element bits 8-9
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] *= 0.03125f;
    } else {
#pragma unroll
        for (int r = 0; r < 16; ++r) tile[17 * t + r] = v[r];
        named_barrier(bar, 64);
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = tile[pad16(256 * (r >> 2) + 4 * t + (r & 3))];
    }
    float mx = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) mx = fmaxf(mx, fabsf(v[r]));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    if (lane == 0) pmax[t >> 5] = mx;
    named_barrier(bar, 64);      // also: every thread has read its tile values
    return fmaxf(pmax[0], pmax[1]);
}

}  // namespace ninfer
