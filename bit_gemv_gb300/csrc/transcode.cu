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
// A 256-entry table in shared memory gives each byte's digits as a 10-bit
// PQ2_0 pattern (digit i at bits 2i, for all 256 byte values by the same
// formula); base byte j's pattern lands at bit 10 j of the group's 256-bit code
// run, high byte h's low 8 bits at bit 240 + 8 h. Each thread rewrites kUnits
// (row, group) units, consecutive threads taking consecutive groups of a row, so
// the 24-byte reads and the 32-byte writes are contiguous across a warp.
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "gemv.h"

namespace ninfer {
namespace {

constexpr int kThreads = 256;
constexpr int kUnits = 4;          // units per thread

struct Planes {
    const uint8_t *base, *high, *scale;     // PTQ1_0 planes
    uint8_t *qbase, *qscale;                // PQ2_0 planes
    uint64_t groups, units;                 // groups per row, rows * groups
};

__global__ void __launch_bounds__(kThreads) ptq1_to_pq2_kernel(const Planes p) {
    __shared__ uint16_t lut[256];
    pdl_launch_dependents();
    {
        uint32_t B = threadIdx.x, c = 0;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            c |= (B % 3) << (2 * i);
            B /= 3;
        }
        lut[threadIdx.x] = (uint16_t)c;
    }
    __syncthreads();
    const uint64_t u0 = (uint64_t)blockIdx.x * (kThreads * kUnits) + threadIdx.x;
    // the payload is a read-only parameter: read it before the dependency wait
    uint32_t bw[kUnits][6], hb[kUnits];
    uint16_t sc[kUnits];
#pragma unroll
    for (int k = 0; k < kUnits; ++k) {
        const uint64_t u = u0 + (uint64_t)k * kThreads;
        const bool live = u < p.units;
        const uint64_t r = live ? u / p.groups : 0, g = live ? u % p.groups : 0;
        const uint2 *src = reinterpret_cast<const uint2 *>(p.base + r * (24 * p.groups) + 24 * g);
        const uint2 b0 = src[0], b1 = src[1], b2 = src[2];
        bw[k][0] = b0.x; bw[k][1] = b0.y; bw[k][2] = b1.x; bw[k][3] = b1.y; bw[k][4] = b2.x; bw[k][5] = b2.y;
        hb[k] = *reinterpret_cast<const uint16_t *>(p.high + r * (2 * p.groups) + 2 * g);
        sc[k] = reinterpret_cast<const uint16_t *>(p.scale)[r * p.groups + g];
    }
    pdl_wait();          // the previous call's GEMM may still read the output buffer
#pragma unroll
    for (int k = 0; k < kUnits; ++k) {
        const uint64_t u = u0 + (uint64_t)k * kThreads;
        if (u >= p.units) break;
        const uint64_t r = u / p.groups, g = u % p.groups;
        uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};      // 16 codes per word, weight j at bits 2 (j % 16)
#pragma unroll
        for (int j = 0; j < 24; ++j) {
            const uint32_t c = lut[(bw[k][j >> 2] >> (8 * (j & 3))) & 0xFFu];
            const int pos = 10 * j, wd = pos >> 5, sh = pos & 31;
            out[wd] |= c << sh;
            if (sh > 22) out[wd + 1] |= c >> (32 - sh);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) out[7] |= ((uint32_t)lut[(hb[k] >> (8 * h)) & 0xFFu] & 0xFFu) << (16 + 8 * h);
        uint4 *dst = reinterpret_cast<uint4 *>(p.qbase + r * (32 * p.groups) + 32 * g);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        // scales: same row-major [n][groups] binary16 layout in both formats
        reinterpret_cast<uint16_t *>(p.qscale)[u] = sc[k];
    }
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
    const uint64_t per_block = (uint64_t)kThreads * kUnits, blocks = (p.units + per_block - 1) / per_block;
    if (blocks > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "PTQ1_0 -> PQ2_0 transcode: too many groups");
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ptq1_to_pq2_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "PTQ1_0 -> PQ2_0 transcode launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
