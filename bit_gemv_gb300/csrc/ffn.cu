// ninfer_ternary_gate_up: the FFN gate and up projections of one activation
// with the SwiGLU product, y = silu(Wg xr_g) * (Wu xr_u).
//
// Fused gate/up weights keep each original projection's transform (TensorSharp
// article §4.2), so xr_g and xr_u are x rotated with the gate's and the up
// projection's signs. The layers' FFN is the dense gated FFN of the Qwen 3.5
// family (same article §4.4), read here as SwiGLU: silu(a) = a / (1 + e^-a).
//
// Decode (PQ2_0, M = 1): one kernel streams the rows of both matrices, keeps
// both sums per row and stores the product (gemv_pq2_int.cu, two-matrix
// instance): one launch, one read of x, no intermediate in memory. Every other
// case runs the two projections through ninfer_ternary_matmul into fp32
// workspace rows and then swiglu_kernel.
#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
int device_info(DeviceInfo *out);

namespace {

__global__ void __launch_bounds__(256) swiglu_kernel(const float *g, const float *u, void *y, int y_dtype,
                                                     uint64_t count) {
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float a = g[i];
    store1(y, i, y_dtype, a / (1.f + expf(-a)) * u[i]);
}

struct FfnPlan {
    bool fused;
    IntPlan gint;
    uint64_t inter_bytes;     // fp32 gate and up rows (general path)
    uint64_t mm_bytes;        // workspace of one ninfer_ternary_matmul call (general path)
    uint64_t workspace;
};

int plan_ffn(int fmt, const ninfer_row_split_geometry &g, uint64_t M, bool rotate, bool distinct_signs, FfnPlan *fp) {
    *fp = FfnPlan{};
    DeviceInfo d;
    int st = device_info(&d);
    if (st) return st;
    if (fmt == NINFER_PQ2_0_G128 && gemv_pq2_int_plan(g, M, rotate, d.sms, d.smem_optin, &fp->gint, 2, distinct_signs)) {
        fp->fused = true;
        return NINFER_OK;
    }
    uint64_t mn;
    if (!mul_ok(M, g.n, &mn) || mn > UINT64_MAX / 16) return fail(NINFER_ERR_OVERFLOW, "gate/up: M * n overflows");
    fp->inter_bytes = (2 * mn * sizeof(float) + 255) / 256 * 256;
    st = ninfer_ternary_matmul_workspace(fmt, g.n, g.k, M, rotate ? 1 : 0, &fp->mm_bytes);
    if (st) return st;
    fp->workspace = fp->inter_bytes + fp->mm_bytes;
    return NINFER_OK;
}

}  // namespace
}  // namespace ninfer

using namespace ninfer;

extern "C" int ninfer_ternary_gate_up_workspace(int fmt, uint64_t n, uint64_t k, uint64_t M, int rotate,
                                                int distinct_signs, uint64_t *bytes) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!bytes) return fail(NINFER_ERR_INVALID_ARGUMENT, "gate/up workspace: NULL output");
    if (M == 0) return fail(NINFER_ERR_SHAPE, "gate/up workspace: M must be positive");
    FfnPlan fp;
    st = plan_ffn(fmt, g, M, rotate != 0, distinct_signs != 0, &fp);
    if (st) return st;
    *bytes = fp.workspace;
    return NINFER_OK;
}

extern "C" int ninfer_ternary_gate_up(int fmt, const uint8_t *payload_gate, const uint8_t *payload_up,
                                      uint64_t payload_bytes, uint64_t n, uint64_t k, const void *x, int x_dtype,
                                      const uint16_t *signs_gate_bf16, const uint16_t *signs_up_bf16, void *y,
                                      int y_dtype, uint64_t M, void *workspace, uint64_t workspace_bytes,
                                      ninfer_stream stream) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!payload_gate || !payload_up || !x || !y)
        return fail(NINFER_ERR_INVALID_ARGUMENT, "gate/up: NULL payload, x or y");
    if (M == 0) return fail(NINFER_ERR_SHAPE, "gate/up: M must be positive");
    if ((signs_gate_bf16 == nullptr) != (signs_up_bf16 == nullptr))
        return fail(NINFER_ERR_INVALID_ARGUMENT, "gate/up: give both sign vectors or neither");
    if (!dtype_valid(x_dtype)) return fail(NINFER_ERR_INVALID_ARGUMENT, "gate/up: x dtype %d unsupported", x_dtype);
    if (y_dtype != NINFER_F32 && y_dtype != NINFER_BF16)
        return fail(NINFER_ERR_INVALID_ARGUMENT, "gate/up: y dtype must be f32 or bf16");
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    auto aligned = [](const void *ptr, uintptr_t a) { return reinterpret_cast<uintptr_t>(ptr) % a == 0; };
    if (!aligned(payload_gate, 256) || !aligned(payload_up, 256))
        return fail(NINFER_ERR_ALIGNMENT, "gate/up: payloads must be 256-byte aligned");
    if (!aligned(x, 16) || !aligned(y, 16)) return fail(NINFER_ERR_ALIGNMENT, "gate/up: x and y must be 16-byte aligned");
    const bool rotate = signs_gate_bf16 != nullptr;
    if (rotate && k % 1024)
        return fail(NINFER_ERR_SHAPE, "gate/up: k=%llu is not a multiple of 1024; the rotated input needs whole blocks",
                    (unsigned long long)k);
    if (rotate && (!aligned(signs_gate_bf16, 16) || !aligned(signs_up_bf16, 16)))
        return fail(NINFER_ERR_ALIGNMENT, "gate/up: signs must be 16-byte aligned");
    FfnPlan fp;
    st = plan_ffn(fmt, g, M, rotate, signs_gate_bf16 != signs_up_bf16, &fp);
    if (st) return st;
    if (fp.workspace && (!workspace || workspace_bytes < fp.workspace))
        return fail(NINFER_ERR_SIZE_MISMATCH, "gate/up: workspace of %llu bytes needed, %llu given",
                    (unsigned long long)fp.workspace, (unsigned long long)workspace_bytes);
    if (fp.workspace && !aligned(workspace, 256))
        return fail(NINFER_ERR_ALIGNMENT, "gate/up: workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fp.fused)
        return gemv_pq2_int_launch(fp.gint, payload_gate, g, x, x_dtype, signs_gate_bf16, y, y_dtype, s,
                                   prefetch_before_dependency(), payload_up, signs_up_bf16);
    float *gate = static_cast<float *>(workspace), *up = gate + M * n;
    uint8_t *mm = static_cast<uint8_t *>(workspace) + fp.inter_bytes;
    st = ninfer_ternary_matmul(fmt, payload_gate, payload_bytes, n, k, x, x_dtype, signs_gate_bf16, gate, NINFER_F32,
                               M, mm, fp.mm_bytes, stream);
    if (st) return st;
    st = ninfer_ternary_matmul(fmt, payload_up, payload_bytes, n, k, x, x_dtype, signs_up_bf16, up, NINFER_F32, M, mm,
                               fp.mm_bytes, stream);
    if (st) return st;
    const uint64_t count = M * n;
    swiglu_kernel<<<(unsigned)((count + 255) / 256), 256, 0, s>>>(gate, up, y, y_dtype, count);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gate/up: SwiGLU launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}
