// ninfer_ternary_matmul: argument checks, workspace sizing and dispatch.
#include <mutex>

#include <cuda_runtime.h>

#include "common.h"
#include "device.cuh"
#include "gemv.h"
#include "plane.cuh"

namespace ninfer {
int gemm_simple_launch(const PlaneView &p, uint64_t n, uint64_t k, const void *a, int a_dtype, uint64_t M, void *y,
                       int y_dtype, cudaStream_t stream);

int device_info(DeviceInfo *out) {
    static DeviceInfo cache[64];
    static bool have[64];
    static std::mutex mu;     // first calls from several host threads
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && have[dev]) {
        *out = cache[dev];
        return NINFER_OK;
    }
    DeviceInfo d{};
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "device attributes: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) {
        cache[dev] = d;
        have[dev] = true;
    }
    *out = d;
    return NINFER_OK;
}

static bool g_pdl = true;
bool prefetch_before_dependency() { return g_pdl; }
}  // namespace ninfer

using namespace ninfer;

namespace {
enum class Path { kIntPq2, kIntPtq1, kMmaPq2, kMmaPtq1, kTcPq2, kTcPtq1, kTiled };

struct MatmulPlan {
    Path path;
    IntPlan gint;
    Ptq1Plan gptq;
    MmaPlan gmma;
    Ptq1MmaPlan gpm;
    TcPlan gtc;
    ninfer_row_split_geometry q;     // PQ2_0 geometry of the transcoded planes (kTcPtq1)
    uint64_t q_bytes;                // their bytes in the workspace, 256-aligned
    uint64_t workspace;
};

int plan_matmul(int fmt, const ninfer_row_split_geometry &g, uint64_t M, bool rotate, MatmulPlan *mp) {
    DeviceInfo d;
    int st = device_info(&d);
    if (st) return st;
    mp->workspace = 0;
    if (fmt == NINFER_PQ2_0_G128 && gemv_pq2_int_plan(g, M, rotate, d.sms, d.smem_optin, &mp->gint)) {
        mp->path = Path::kIntPq2;
        mp->workspace = mp->gint.workspace;     // none: each CTA rotates x itself
        return NINFER_OK;
    }
    if (fmt == NINFER_PTQ1_0_G128 && gemv_ptq1_int_plan(g, M, rotate, d.sms, d.smem_optin, &mp->gptq)) {
        mp->path = Path::kIntPtq1;
        mp->workspace = mp->gptq.workspace;     // none: the CTAs rotate x themselves
        return NINFER_OK;
    }
    if (fmt == NINFER_PQ2_0_G128 && gemv_pq2_mma_plan(g, M, rotate, d.sms, d.smem_optin, &mp->gmma)) {
        mp->path = Path::kMmaPq2;
        mp->workspace = mp->gmma.workspace;     // the activation fragments
        return NINFER_OK;
    }
    if (fmt == NINFER_PTQ1_0_G128 && gemv_ptq1_mma_plan(g, M, rotate, d.sms, d.smem_optin, &mp->gpm)) {
        mp->path = Path::kMmaPtq1;
        mp->workspace = mp->gpm.workspace;      // per-block partial sums
        return NINFER_OK;
    }
    if (fmt == NINFER_PQ2_0_G128 && gemm_tc_plan(g, M, d.sms, d.smem_optin, &mp->gtc)) {
        mp->path = Path::kTcPq2;
        mp->workspace = mp->gtc.workspace;     // xr as binary16
        return NINFER_OK;
    }
    if (fmt == NINFER_PTQ1_0_G128 && M > 8 && geometry(NINFER_PQ2_0_G128, g.n, g.k, &mp->q) == NINFER_OK &&
        gemm_tc_plan(mp->q, M, d.sms, d.smem_optin, &mp->gtc)) {
        // prefill: the planes are rewritten as PQ2_0 planes in the workspace, then the
        // same tensor-core GEMM runs on them
        mp->path = Path::kTcPtq1;
        mp->q_bytes = (mp->q.payload_bytes + 255) / 256 * 256;
        mp->workspace = mp->q_bytes + mp->gtc.workspace;
        return NINFER_OK;
    }
    mp->path = Path::kTiled;
    mp->workspace = rotate ? M * g.k * sizeof(float) : 0;   // rotated activations, fp32
    return NINFER_OK;
}
}  // namespace

extern "C" int ninfer_set_prefetch_before_dependency(int enable) {
    g_pdl = enable != 0;
    return NINFER_OK;
}

extern "C" int ninfer_ternary_matmul_workspace(int fmt, uint64_t n, uint64_t k, uint64_t M, int rotate,
                                               uint64_t *bytes) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!bytes) return fail(NINFER_ERR_INVALID_ARGUMENT, "workspace: NULL output");
    if (M == 0) return fail(NINFER_ERR_SHAPE, "workspace: M must be positive");
    uint64_t mk;
    if (!mul_ok(M, k, &mk) || mk > (UINT64_MAX / 8)) return fail(NINFER_ERR_OVERFLOW, "workspace size overflows");
    MatmulPlan mp;
    st = plan_matmul(fmt, g, M, rotate != 0, &mp);
    if (st) return st;
    *bytes = mp.workspace;
    return NINFER_OK;
}

extern "C" int ninfer_ternary_matmul(int fmt, const uint8_t *payload, uint64_t payload_bytes, uint64_t n, uint64_t k,
                                     const void *x, int x_dtype, const uint16_t *signs_bf16, void *y, int y_dtype,
                                     uint64_t M, void *workspace, uint64_t workspace_bytes, ninfer_stream stream) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!payload || !x || !y) return fail(NINFER_ERR_INVALID_ARGUMENT, "matmul: NULL payload, x or y");
    if (M == 0) return fail(NINFER_ERR_SHAPE, "matmul: M must be positive");
    if (!dtype_valid(x_dtype)) return fail(NINFER_ERR_INVALID_ARGUMENT, "matmul: x dtype %d unsupported", x_dtype);
    if (y_dtype != NINFER_F32 && y_dtype != NINFER_BF16)
        return fail(NINFER_ERR_INVALID_ARGUMENT, "matmul: y dtype must be f32 or bf16");
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    if (!aligned(payload, 256)) return fail(NINFER_ERR_ALIGNMENT, "matmul: payload must be 256-byte aligned");
    if (!aligned(x, 16) || !aligned(y, 16)) return fail(NINFER_ERR_ALIGNMENT, "matmul: x and y must be 16-byte aligned");
    const bool rotate = signs_bf16 != nullptr;
    if (rotate && k % 1024)
        return fail(NINFER_ERR_SHAPE, "matmul: k=%llu is not a multiple of 1024; the rotated input needs whole blocks",
                    (unsigned long long)k);
    if (rotate && !aligned(signs_bf16, 16)) return fail(NINFER_ERR_ALIGNMENT, "matmul: signs must be 16-byte aligned");
    MatmulPlan mp;
    st = plan_matmul(fmt, g, M, rotate, &mp);
    if (st) return st;
    const uint64_t need = mp.workspace;
    if (need && (!workspace || workspace_bytes < need))
        return fail(NINFER_ERR_SIZE_MISMATCH, "matmul: workspace of %llu bytes needed, %llu given",
                    (unsigned long long)need, (unsigned long long)workspace_bytes);
    if (need && !aligned(workspace, 16)) return fail(NINFER_ERR_ALIGNMENT, "matmul: workspace must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (mp.path == Path::kIntPq2)
        return gemv_pq2_int_launch(mp.gint, payload, g, x, x_dtype, signs_bf16, y, y_dtype, s, g_pdl);
    if (mp.path == Path::kIntPtq1)
        return gemv_ptq1_int_launch(mp.gptq, payload, g, x, x_dtype, signs_bf16, y, y_dtype, workspace, s, g_pdl);
    if (mp.path == Path::kMmaPq2)
        return gemv_pq2_mma_launch(mp.gmma, payload, g, x, x_dtype, signs_bf16, y, y_dtype, M, workspace, s, g_pdl);
    if (mp.path == Path::kMmaPtq1)
        return gemv_ptq1_mma_launch(mp.gpm, payload, g, x, x_dtype, signs_bf16, y, y_dtype, M, workspace, s, g_pdl);
    if (mp.path == Path::kTcPq2)
        return gemm_tc_launch(mp.gtc, payload, g, x, x_dtype, signs_bf16, y, y_dtype, M, workspace, s);
    if (mp.path == Path::kTcPtq1) {
        uint8_t *qp = static_cast<uint8_t *>(workspace);
        st = ptq1_to_pq2_launch(payload, g, qp, mp.q, s, g_pdl);
        if (st) return st;
        return gemm_tc_launch(mp.gtc, qp, mp.q, x, x_dtype, signs_bf16, y, y_dtype, M, qp + mp.q_bytes, s);
    }
    const PlaneView p = make_view(payload, g, fmt);
    const void *a = x;
    int a_dtype = x_dtype;
    if (rotate) {
        st = ninfer_hadamard_fwd(x, x_dtype, workspace, NINFER_F32, signs_bf16, M, k, stream);
        if (st) return st;
        a = workspace;
        a_dtype = NINFER_F32;
    }
    return gemm_simple_launch(p, n, k, a, a_dtype, M, y, y_dtype, s);
}
