// PTQ1_0_G128 planes -> PQ2_0_G128 planes, on the device, for the prefill path.
//
// Both formats store the same ternary values as offset codes t = value + 1
// ("bonsai三元GGUF模型转ninfer模型01" §3-§4; "GGUF 完整讲解" §4.3): PTQ1_0 packs
// them as base-3 digits (base byte j of a group holds weights 5j .. 5j+4 as
// (byte / 3^i) % 3, high byte h holds weights 120 + 4h .. 123 + 4h), PQ2_0 as
// 2-bit fields (weight j of a group at bits 2 (j % 4) of byte j / 4). The
// scales are the same binary16 values. Rewriting the codes is therefore exact,
// and the tensor-core GEMM, whose weight expansion is written for 2-bit codes,
// serves PTQ1_0 unchanged: one pass over the 28 bytes of every group, writing
// 34, costs a few microseconds against hundreds for the GEMM.
//
// One thread per (row, group); consecutive threads take consecutive groups of
// a row, so both the 24-byte reads and the 32-byte writes are contiguous.
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "gemv.h"

namespace ninfer {
namespace {

struct Planes {
    const uint8_t *base, *high, *scale;     // PTQ1_0 planes
    uint8_t *qbase, *qscale;                // PQ2_0 planes
    uint64_t groups, units;                 // groups per row, rows * groups
};

__global__ void __launch_bounds__(256) ptq1_to_pq2_kernel(const Planes p) {
    pdl_launch_dependents();
    const uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = u < p.units;
    const uint64_t r = live ? u / p.groups : 0, g = live ? u % p.groups : 0;
    // the payload is a read-only parameter: read it before the dependency wait
    const uint2 *src = reinterpret_cast<const uint2 *>(p.base + r * (24 * p.groups) + 24 * g);
    const uint2 b0 = src[0], b1 = src[1], b2 = src[2];
    const uint32_t bw[6] = {b0.x, b0.y, b1.x, b1.y, b2.x, b2.y};
    const uint32_t hb = *reinterpret_cast<const uint16_t *>(p.high + r * (2 * p.groups) + 2 * g);
    const uint16_t sc = reinterpret_cast<const uint16_t *>(p.scale)[r * p.groups + g];
    pdl_wait();          // the previous call's GEMM may still read the output buffer
    if (!live) return;
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};      // 16 codes per word, weight j at bits 2 (j % 16)
#pragma unroll
    for (int j = 0; j < 26; ++j) {
        uint32_t B = j < 24 ? (bw[j >> 2] >> (8 * (j & 3))) & 0xFFu : (hb >> (8 * (j - 24))) & 0xFFu;
        const int nd = j < 24 ? 5 : 4, w0 = j < 24 ? 5 * j : 120 + 4 * (j - 24);
#pragma unroll
        for (int i = 0; i < nd; ++i) {
            const uint32_t t = B % 3;
            B /= 3;
            const int w = w0 + i;
            out[w >> 4] |= t << (2 * (w & 15));
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(p.qbase + r * (32 * p.groups) + 32 * g);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    // scales: same row-major [n][groups] binary16 layout in both formats
    reinterpret_cast<uint16_t *>(p.qscale)[u] = sc;
}

}  // namespace

int ptq1_to_pq2_launch(const uint8_t *payload, const ninfer_row_split_geometry &g, uint8_t *out,
                       const ninfer_row_split_geometry &q, cudaStream_t stream, bool pdl) {
    Planes p;
    p.base = payload + g.base_offset;
    p.high = payload + g.high_offset;
    p.scale = payload + g.scale_offset;
    p.qbase = out + q.base_offset;
    p.qscale = out + q.scale_offset;
    p.groups = g.groups_per_row;
    p.units = g.n * g.groups_per_row;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.units + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ptq1_to_pq2_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "PTQ1_0 -> PQ2_0 transcode launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
