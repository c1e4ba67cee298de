// Device-side view of a row-split payload ("bonsai三元GGUF模型转ninfer模型01"
// §3): base plane at base_offset, high plane at high_offset, scale plane at
// scale_offset, each row-major [row][group][bytes].
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ninfer_ternary.h"

namespace ninfer {

struct PlaneView {
    const uint8_t *base;   // payload + base_offset
    const uint8_t *high;   // payload + high_offset
    const uint8_t *scale;  // payload + scale_offset
    uint64_t base_row, high_row, scale_row;  // bytes per row in each plane
    uint32_t groups;                         // groups per row
    int fmt;
};

inline PlaneView make_view(const uint8_t *payload, const ninfer_row_split_geometry &g, int fmt) {
    PlaneView v;
    v.base = payload + g.base_offset;
    v.high = payload + g.high_offset;
    v.scale = payload + g.scale_offset;
    v.base_row = g.base_row_bytes;
    v.high_row = g.high_row_bytes;
    v.scale_row = g.scale_row_bytes;
    v.groups = (uint32_t)g.groups_per_row;
    v.fmt = fmt;
    return v;
}

// Ternary value (code - 1) of weight j (< 128) of group gi of row r.
// PQ2_0: 2-bit field j % 4 of byte j / 4, least significant first ("GGUF 完整讲解"
// §4.3); code 3 reads +2. PTQ1_0: base-3 digit j % 5 of base byte j / 5 for
// j < 120, digit (j - 120) % 4 of high byte (j - 120) / 4 otherwise.
__device__ __forceinline__ int plane_value(const PlaneView &p, uint64_t r, uint32_t gi, int j) {
    if (p.fmt == NINFER_PQ2_0_G128) {
        const uint8_t b = p.base[r * p.base_row + (uint64_t)gi * 32 + (j >> 2)];
        return (int)((b >> (2 * (j & 3))) & 3) - 1;
    }
    uint32_t b, d;
    if (j < 120) {
        b = p.base[r * p.base_row + (uint64_t)gi * 24 + j / 5];
        d = j % 5;
    } else {
        b = p.high[r * p.high_row + (uint64_t)gi * 2 + (j - 120) / 4];
        d = (j - 120) % 4;
    }
    for (uint32_t i = 0; i < d; ++i) b /= 3;
    return (int)(b % 3) - 1;
}

__device__ __forceinline__ float plane_scale(const PlaneView &p, uint64_t r, uint32_t gi) {
    const uint8_t *s = p.scale + r * p.scale_row + 2ull * gi;
    return __half2float(__ushort_as_half((uint16_t)(s[0] | (s[1] << 8))));
}

}  // namespace ninfer
