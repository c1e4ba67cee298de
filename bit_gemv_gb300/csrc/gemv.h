// Launch plans of the fused decode kernels (shared by matmul.cu and the kernels).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ninfer_ternary.h"

namespace ninfer {


// Device properties the plans depend on (queried once per device).
struct DeviceInfo {
    int sms;
    int smem_optin;
};
int device_info(DeviceInfo *out);
// Device address of the library's error word on the current device.
int device_error_word(uint32_t **out);
// Whether decode kernels may request weights before the dependency wait
// (ninfer_set_prefetch_before_dependency).
bool prefetch_before_dependency();
// Bound, in SM clock cycles, of the weight-ring waits of the kernels that take
// it as a parameter (ninfer_set_wait_limit; default about two seconds).
long long wait_limit_cycles();
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel, device and size.
int set_smem_attribute(const void *kernel, int bytes);

// Rows of a plane as a 2-D byte tensor {row_bytes, rows}, for 2-D box loads:
// boxes of box_bytes x box_rows, optionally 128-byte swizzled.
int encode_rows(CUtensorMap *map, const uint8_t *addr, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                uint32_t box_rows, bool swizzle128);
// Equal row ranges of a plane as a 3-D byte tensor {row_bytes, rows, tiles},
// for 3-D box loads (always rank 3, also for a single tile), so that a box never
// reads past the end of its own range.
int encode_row_tiles(CUtensorMap *map, const uint8_t *addr, uint64_t row_bytes, uint64_t rows, uint64_t tiles,
                     uint32_t box_bytes, uint32_t box_rows, bool swizzle128);

// A 3-D tensor of 8-byte elements (dims[0] contiguous; strides in bytes of
// dims 1-2), unswizzled boxes of box[0] x box[1] x box[2] elements.
int encode_3d_u64(CUtensorMap *map, const uint8_t *addr, const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                  const uint32_t (&box)[3]);

// A 2-D tensor map over a row-major array: `inner` elements per row, `outer`
// rows, rows `row_stride_bytes` apart; boxes of box_inner x box_outer.
int encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *addr, uint64_t inner,
              uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

// M = 1 integer kernel (PQ2_0_G128), rotation fused in. With mats = 2 it
// streams two matrices of the same geometry (FFN gate and up) for the same rows
// and stores silu(gate x) * (up x); two_rotations when their signs differ.
struct IntPlan {
    bool ok;
    int mats;
    uint32_t act_one;
    uint32_t grid, grid_rows, rows_per_cta, nitem, nslots, pre_issue, nrot;
    bool cluster;                // CTA pairs share the rotations (grid even)
    uint32_t off_ring, off_act, off_rot, off_part, off_bar, off_cnt, smem;
    uint64_t workspace;
};
bool gemv_pq2_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                       IntPlan *plan, int mats = 1, bool two_rotations = false);
int gemv_pq2_int_launch(const IntPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                        int x_dtype, const uint16_t *signs, void *y, int y_dtype, cudaStream_t stream, bool pdl,
                        const uint8_t *payload2 = nullptr, const uint16_t *signs2 = nullptr);


// M = 1 integer kernel (PTQ1_0_G128), rotation fused in.
struct Ptq1Plan {
    bool ok;
    uint32_t cluster;        // CTAs of a cluster, which split the groups of one row range (1: none)
    uint32_t grid, units, rows_per_cta, ng, hbytes, wg, nbx, bstride, nsets, u, nslots, pre_issue;
    uint32_t slot_bytes, slot_high, slot_scale, part_stride, part_slot_bytes;
    uint32_t off_ring, off_part, off_rs, off_bar, smem;
    uint64_t workspace;
};
bool gemv_ptq1_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                        Ptq1Plan *plan);
int gemv_ptq1_int_launch(const Ptq1Plan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, void *workspace,
                         cudaStream_t stream, bool pdl);

// 2 <= M <= 8, PQ2_0_G128: binary16 mma.sync kernel with a prep kernel for the fragments.
struct MmaPlan {
    bool ok;
    uint32_t grid, rows_per_cta, nitem, nslots, pre_issue, fx_bytes;
    uint32_t off_ring, off_frag, off_fx, off_acc, off_part, off_bar, off_cnt, smem;
    uint64_t workspace;
};
bool gemv_pq2_mma_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                       MmaPlan *plan);
int gemv_pq2_mma_launch(const MmaPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                        int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, void *workspace,
                        cudaStream_t stream, bool pdl);

// 1 <= M <= 8, PTQ1_0_G128: binary16 mma.sync kernel split over the 1024-blocks
// of k, plus a reduction kernel over the blocks (gemv_ptq1_mma.cu).
struct Ptq1MmaPlan {
    bool ok;
    uint32_t nblk, tiles, rows_per_tile, nslots;
    uint32_t off_ring, off_lut, off_rot, off_frag, off_bar, off_cnt, smem;
    uint64_t n_pad;
    uint64_t workspace;
};
bool gemv_ptq1_mma_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                        Ptq1MmaPlan *plan);
int gemv_ptq1_mma_launch(const Ptq1MmaPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M,
                         void *workspace, cudaStream_t stream, bool pdl);

// PTQ1_0 planes rewritten exactly as PQ2_0 planes (transcode.cu), for the prefill path.
int ptq1_to_pq2_launch(const uint8_t *payload, const ninfer_row_split_geometry &g, uint8_t *out,
                       const ninfer_row_split_geometry &q, cudaStream_t stream, bool pdl);

// Prefill (M > 8) tensor-core path for PQ2_0_G128 (gemm_tc.cu).
struct TcPlan {
    bool ok;
    uint32_t grid_n, grid_m, grid, smem;     // weight tiles, token tiles, persistent CTAs
    uint64_t workspace;
};
bool gemm_tc_plan(const ninfer_row_split_geometry &g, uint64_t M, int sms, int smem_limit, TcPlan *plan);
int gemm_tc_launch(const TcPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                   int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, void *workspace,
                   cudaStream_t stream);

}  // namespace ninfer
