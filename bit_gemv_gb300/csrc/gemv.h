// Launch plans of the fused decode kernels (shared by matmul.cu and the kernels).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ninfer_ternary.h"

namespace ninfer {

struct GemvPlan {
    bool ok;
    uint32_t grid, rows_per_cta, nbox, nt, nslots, slot_bytes;
    uint32_t off_b, off_fo, off_red, off_bar, smem;
};

// Device properties the plans depend on (queried once per device).
struct DeviceInfo {
    int sms;
    int smem_optin;
};
int device_info(DeviceInfo *out);
// Device address of the library's error word on the current device.
int device_error_word(uint32_t **out);

bool gemv_pq2_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                   GemvPlan *plan);
int gemv_pq2_launch(const GemvPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                    int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, cudaStream_t stream,
                    bool pdl);

}  // namespace ninfer
