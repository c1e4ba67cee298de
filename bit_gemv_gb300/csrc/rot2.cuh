// Rotation of one 1024-element block of the activation by a pair of warps,
// shared by the M = 1 decode kernels: the forward signed block Walsh-Hadamard
// transform ("artifact-container.md" §8 hadamard_signs; TensorSharp article
// §4.2: per 1024-block H (D * x) / 32) and rounding to 16-bit fixed point,
// x16 = rint(xr * 2^E') with E' chosen per block so that max |x16| < 2^14.
#pragma once

#include <cstdint>

#include "async.cuh"
#include "device.cuh"

namespace ninfer {

constexpr uint32_t kRotScratchBytes = 4352;     // per rotating pair: 1080 + 2 floats

// The two warps of a pair rotate one 1024-element block together; thread
// t = lane + 32 wh of the pair. Layout A (the load layout): v[8i + r] = element
// 512 i + 8 t + r (i < 2, r < 8). Zero past k.
template <int kXType>
__device__ __forceinline__ void load_block2(const void *x, uint32_t k, uint32_t b, int t, float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float u[8];
        const uint64_t idx = (uint64_t)b * 1024 + 512 * i + 8 * t;
        if (idx + 8 <= k) {
            load8(x, idx, kXType, u);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = idx + e < k ? load1(x, idx + e, kXType) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * i + e] = u[e];
    }
}

__device__ __forceinline__ void load_signs2(const uint16_t *s, uint32_t b, int t, float (&d)[16]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float u[8];
        load_signs8(s, (uint64_t)b * 1024 + 512 * i + 8 * t, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) d[8 * i + e] = u[e];
    }
}

__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void f2unpack(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// Butterflies over the four register index bits of 16 values: bits 1-3 as
// paired fp32 adds and subtracts (each element rounded exactly as by a scalar
// add), bit 0 within the pairs.
__device__ __forceinline__ void butterfly16_f32x2(float (&v)[16]) {
    uint64_t w[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) w[m] = f2pack(v[2 * m], v[2 * m + 1]);
#pragma unroll
    for (int bit = 0; bit < 3; ++bit)
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            if (m & (1 << bit)) continue;
            uint64_t sum, dif;
            asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(w[m]), "l"(w[m | (1 << bit)]));
            asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(w[m]), "l"(w[m | (1 << bit)]));
            w[m] = sum;
            w[m | (1 << bit)] = dif;
        }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        float a, c;
        f2unpack(w[m], a, c);
        v[2 * m] = a + c;
        v[2 * m + 1] = a - c;
    }
}

// Rotates block b with the pair (x in v as load_block2 leaves it; signs in d
// unless rotate is false) and rounds it to 16-bit fixed point. Stages:
// register butterflies on element bits {0,1,2,9} (layout A); a transpose
// through the pair's scratch to layout B (lane = element bits {0,1,2,7,8},
// wh = bit 9, register j = bits 3-6: e = (lane & 7) + 8 j + 128 (lane >> 3) +
// 512 wh) for register butterflies on bits 3-6 and two shuffle stages on bits
// 7-8; a transpose back to layout A, where each thread again holds the runs
// of eight consecutive elements 512 i + 8 t .. + 7 (i < 2). Scratch slot of
// element e: e + 8 (e >> 7); the pair's maximum goes through floats 1080-1081.
// On return qb[8 i + r] holds, in its low 16 bits, x16 of element 512 i + 8 t + r
// (the bits minus 0x4B400000 are x16 as an int), and the return value is E,
// x16 = rint(v * 2^E) for the unnormalised v = H (D x) = 32 xr (rotate) or v = x.
// bar: the pair's named barrier. The scratch may be reused on return.
__device__ __forceinline__ int rotate_quant2(bool rotate, float (&v)[16], const float (&d)[16], float *scr, int t,
                                             uint32_t bar, uint32_t (&qb)[16]) {
    const int lane = t & 31, wh = t >> 5;
    if (rotate) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            uint64_t r;
            asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2pack(v[2 * m], v[2 * m + 1])),
                "l"(f2pack(d[2 * m], d[2 * m + 1])));
            f2unpack(r, v[2 * m], v[2 * m + 1]);
        }
        butterfly16_f32x2(v);      // element bits 0, 1, 2, 9
    }
    const int aA = 8 * t + 8 * (t >> 4);
    const int aB = (lane & 7) + 136 * (lane >> 3) + 544 * wh;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 2; ++c)
            *reinterpret_cast<float4 *>(scr + 544 * i + aA + 4 * c) =
                make_float4(v[8 * i + 4 * c], v[8 * i + 4 * c + 1], v[8 * i + 4 * c + 2], v[8 * i + 4 * c + 3]);
    named_barrier(bar, 64);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = scr[aB + 8 * j];
    if (rotate) {
        butterfly16_f32x2(v);      // element bits 3-6
        // element bits 7 and 8 (lane bits 3 and 4): the lane whose bit is set keeps
        // partner - own, the other own + partner (fmaf(+-1, own, partner): one rounding)
#pragma unroll
        for (int s = 8; s <= 16; s <<= 1) {
            const float sg = (lane & s) ? -1.f : 1.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = fmaf(sg, v[j], __shfl_xor_sync(0xffffffffu, v[j], s));
        }
    }
    // each thread rewrites exactly the slots it read, so only the reads below wait
#pragma unroll
    for (int j = 0; j < 16; ++j) scr[aB + 8 * j] = v[j];
    named_barrier(bar, 64);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float4 q = *reinterpret_cast<const float4 *>(scr + 544 * i + aA + 4 * c);
            v[8 * i + 4 * c] = q.x;
            v[8 * i + 4 * c + 1] = q.y;
            v[8 * i + 4 * c + 2] = q.z;
            v[8 * i + 4 * c + 3] = q.w;
        }
    // block maximum: a tree in registers, the warp (a non-negative float's bits
    // order as its value: one warp-wide integer max), then the pair
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = fmaxf(fabsf(v[j]), fabsf(v[j + 8]));
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
    float mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m[0])));
    if (lane == 0) scr[1080 + wh] = mx;
    named_barrier(bar, 64);
    mx = fmaxf(scr[1080], scr[1081]);
    int E = 0;
    if (mx > 0.f) E = 13 - ilogbf(mx);     // max |x16| < 2^14
    E = max(-100, min(100, E));
    const float up = ldexpf(1.f, E);
    // x16 = rint(v * 2^E): fma(v, 2^E, 1.5 * 2^23) rounds to nearest (ties to even)
    // and leaves x16 in the low 16 bits
    const uint64_t up2 = f2pack(up, up), mg = f2pack(12582912.0f, 12582912.0f);
#pragma unroll
    for (int m2 = 0; m2 < 8; ++m2) {
        uint64_t r;
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2pack(v[2 * m2], v[2 * m2 + 1])), "l"(up2), "l"(mg));
        float a, c;
        f2unpack(r, a, c);
        qb[2 * m2] = __float_as_uint(a);
        qb[2 * m2 + 1] = __float_as_uint(c);
    }
    named_barrier(bar, 64);      // every thread has read the pair's maximum: the scratch is free
    return E;
}

}  // namespace ninfer
