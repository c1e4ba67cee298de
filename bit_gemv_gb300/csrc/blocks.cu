// Device-side conversion between the ggml stream of single-group blocks and the
// row-split planes ("bonsai三元GGUF模型转ninfer模型01" §3-§4, the block slices
// of assemble_ternary): a model loaded as a block stream into device memory is
// laid out as planes without a trip through the host.
//
// Block layouts: PQ2_0 34 bytes [scale 2][base 32]; PTQ1_0 28 bytes
// [base 24][high 2][scale 2]. Group g of row r is block r * groups_per_row + g;
// its slices go to base_offset + r * base_row_bytes + g * base_bytes_per_group
// (and the same for high and scale). Bytes are moved, never changed, so the two
// directions are exact inverses; the alignment gaps between planes are zero.
//
// One thread per block. The slices sit at 2-byte offsets inside 34-byte blocks,
// so the copies go 16 bits at a time.
#include <cuda_runtime.h>

#include "common.h"
#include "gemv.h"

namespace ninfer {
namespace {

struct BlockMap {
    uint8_t *blocks, *payload;
    uint64_t units, groups, block_bytes;
    uint64_t base_offset, base_row, high_offset, high_row, scale_offset, scale_row;
    uint32_t bs, bl, hs, hl, ss;     // slice offsets and lengths inside a block
};

template <bool kToPlanes>
__global__ void __launch_bounds__(256) block_plane_kernel(const BlockMap p) {
    const uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= p.units) return;
    const uint64_t r = u / p.groups, g = u % p.groups;
    uint16_t *blk = reinterpret_cast<uint16_t *>(p.blocks + u * p.block_bytes);
    uint16_t *base = reinterpret_cast<uint16_t *>(p.payload + p.base_offset + r * p.base_row + g * p.bl);
    uint16_t *scale = reinterpret_cast<uint16_t *>(p.payload + p.scale_offset + r * p.scale_row + 2 * g);
    for (uint32_t i = 0; i < p.bl / 2; ++i) {
        if (kToPlanes) base[i] = blk[p.bs / 2 + i];
        else blk[p.bs / 2 + i] = base[i];
    }
    if (p.hl) {
        uint16_t *high = reinterpret_cast<uint16_t *>(p.payload + p.high_offset + r * p.high_row + g * p.hl);
        if (kToPlanes) high[0] = blk[p.hs / 2];
        else blk[p.hs / 2] = high[0];
    }
    if (kToPlanes) scale[0] = blk[p.ss / 2];
    else blk[p.ss / 2] = scale[0];
}

int convert(bool to_planes, int fmt, uint64_t n, uint64_t k, const uint8_t *blocks, uint64_t blocks_bytes,
            uint8_t *payload, uint64_t payload_bytes, ninfer_stream stream) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!blocks || !payload) return fail(NINFER_ERR_INVALID_ARGUMENT, "device block conversion: NULL buffer");
    const uint64_t nb = fmt == NINFER_PQ2_0_G128 ? 34 : 28, units = n * g.groups_per_row;
    uint64_t want;
    if (!mul_ok(units, nb, &want)) return fail(NINFER_ERR_OVERFLOW, "block stream size overflows");
    if (blocks_bytes != want)
        return fail(NINFER_ERR_SIZE_MISMATCH, "block stream holds %llu bytes; shape requires %llu",
                    (unsigned long long)blocks_bytes, (unsigned long long)want);
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    if (reinterpret_cast<uintptr_t>(blocks) % 2 || reinterpret_cast<uintptr_t>(payload) % 256)
        return fail(NINFER_ERR_ALIGNMENT, "device block conversion: blocks must be 2-byte and payload 256-byte aligned");
    BlockMap p;
    p.blocks = const_cast<uint8_t *>(blocks);
    p.payload = payload;
    p.units = units;
    p.groups = g.groups_per_row;
    p.block_bytes = nb;
    p.base_offset = g.base_offset;
    p.base_row = g.base_row_bytes;
    p.high_offset = g.high_offset;
    p.high_row = g.high_row_bytes;
    p.scale_offset = g.scale_offset;
    p.scale_row = g.scale_row_bytes;
    if (fmt == NINFER_PQ2_0_G128) {
        p.bs = 2; p.bl = 32; p.hs = 0; p.hl = 0; p.ss = 0;
    } else {
        p.bs = 0; p.bl = 24; p.hs = 24; p.hl = 2; p.ss = 26;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (to_planes) e = cudaMemsetAsync(payload, 0, payload_bytes, s);     // the gaps between planes
    if (e == cudaSuccess && units) {
        const dim3 grid((unsigned)((units + 255) / 256));
        if (to_planes) block_plane_kernel<true><<<grid, 256, 0, s>>>(p);
        else block_plane_kernel<false><<<grid, 256, 0, s>>>(p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "device block conversion: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace
}  // namespace ninfer

extern "C" int ninfer_blocks_to_planes_device(int fmt, uint64_t n, uint64_t k, const uint8_t *blocks,
                                              uint64_t blocks_bytes, uint8_t *payload, uint64_t payload_bytes,
                                              ninfer_stream stream) {
    return ninfer::convert(true, fmt, n, k, blocks, blocks_bytes, payload, payload_bytes, stream);
}

extern "C" int ninfer_planes_to_blocks_device(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                                              uint64_t payload_bytes, uint8_t *blocks, uint64_t blocks_bytes,
                                              ninfer_stream stream) {
    return ninfer::convert(false, fmt, n, k, blocks, blocks_bytes, const_cast<uint8_t *>(payload), payload_bytes,
                           stream);
}
