// Decode GEMV for PQ2_0_G128 weights and one activation row (M = 1), on the
// CUDA cores' integer pipes.
//
// What it computes:
//   y[r] = sum_g scale[r][g] * sum_{j<128} (code[r][128g+j] - 1) * xr[128g+j]
// with xr the forward-rotated activation ("artifact-container.md" §8
// hadamard_signs; TensorSharp article §4.2), codes the 2-bit fields of the base
// plane, least significant first, value = code - 1 ("GGUF 完整讲解" §4.3), and
// one binary16 scale per 128-weight group at scale_offset
// ("bonsai三元GGUF模型转ninfer模型01" §3).
//
// Arithmetic: the activation arrives prepared by act_prep.cu as 16-bit fixed
// point per 1024-block (x16 = rint(xr * 2^E)). In a 32-bit word of codes (16
// weights, four per byte) the mask 0x03 << 2p per byte leaves the four codes of
// position p as bytes (times 4^p); dp2a multiplies two of them by two int16
// activations and accumulates exactly in int32. Per group:
//   sum_j c_j x16_j = acc0 + acc1/4 + acc2/16 + acc3/64        (exact shifts)
//   y += scale * 2^-E * (that - sum_j x16_j)                     (value = code - 1)
// GB300 issues LOP3 and dp2a at 64 lanes/clk/SM each (partly co-issuing);
// with two rows per lane the loop sustains ~100 weights/clk/SM, above the
// HBM rate of ~70-80 weights/clk/SM, while legacy mma.sync with changing
// operands reaches only ~55.
//
// Data movement: two CTAs per SM, each owning a contiguous row range. Weights
// stream through a ring of item slots; an item is 64 rows x 4 groups: two
// 128-byte-swizzled tensor boxes of 32 rows x 128 bytes (a 3-D map view keeps
// them inside the CTA's rows) plus the two matching boxes of scales (32 rows x
// 16 bytes). Each item completes on its own mbarrier. The last of the four
// warps reading an item re-arms its slot with the item nslots further on. A
// few items are requested before the programmatic-dependent-launch wait
// (weights are read-only parameters); the prepared activation follows as one
// bulk copy right after the wait, ahead of the rest of the ring.
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
namespace {

constexpr int kThreads = 256;     // 8 warps; two CTAs per SM
constexpr int kWarps = 8;
constexpr int kRows = 64;         // rows per tile: two 32-row boxes, two rows per lane
constexpr uint32_t kItemBytes = 2 * 4096 + 2 * 512;
constexpr uint32_t kMaxSlots = 12;
constexpr uint32_t kActCopies = 8;     // prepared-activation copies, read by CTA % 8

struct IntParams {
    CUtensorMap wmap_main, wmap_last;   // base rows: {row bytes, R rows, CTA} / last CTA {row bytes, rows}
    CUtensorMap smap_main, smap_last;   // scale rows, same views
    const uint8_t *act;                 // prepared activation (act_prep.cu layout), kActCopies copies
    uint64_t act_copy_stride;
    void *y;
    uint64_t n;
    uint32_t groups, nbox, rows_per_cta;
    int y_dtype;
    uint32_t nslots, pre_issue, act_bytes;
    uint32_t off_ring, off_act, off_part, off_bar, off_cnt;
    uint32_t *err;
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

// Item i = tile * nbox + column: its two weight boxes and two scale boxes into
// ring slot i % nslots (one thread).
__device__ __forceinline__ void issue_item(const IntParams &p, uint8_t *smem, uint32_t item, bool last_cta) {
    const uint32_t tile = item / p.nbox, col = item % p.nbox, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kItemBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kItemBytes);
    const int x = (int)(col * 128), xs = (int)((col >> 1) * 16), y0 = (int)(tile * kRows);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (last_cta) {
            tma_load_2d(dst + h * 4096, &p.wmap_last, x, y0 + 32 * h, bar);
            tma_load_2d(dst + 8192 + h * 512, &p.smap_last, xs, y0 + 32 * h, bar);
        } else {
            tma_load_3d(dst + h * 4096, &p.wmap_main, x, y0 + 32 * h, (int)blockIdx.x, bar);
            tma_load_3d(dst + 8192 + h * 512, &p.smap_main, xs, y0 + 32 * h, (int)blockIdx.x, bar);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) gemv_pq2_int_kernel(const __grid_constant__ IntParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t r_begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t r_end = r_begin + p.rows_per_cta < p.n ? r_begin + p.rows_per_cta : p.n;
    const bool last_cta = blockIdx.x == gridDim.x - 1;
    const uint32_t ntile = (uint32_t)((r_end - r_begin + kRows - 1) / kRows);
    const uint32_t nitems = ntile * p.nbox;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t act_bar = bar0 + 8 * kMaxSlots;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);

    if (tid == 0) {
        prefetch_tmap(last_cta ? &p.wmap_last : &p.wmap_main);
        prefetch_tmap(last_cta ? &p.smap_last : &p.smap_main);
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        mbar_init(act_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    if (tid == 0) {
        // weights are read-only parameters: start their stream before waiting
        // on the preceding kernels
        for (uint32_t i = 0; i < p.pre_issue && i < ring_to; ++i) issue_item(p, smem, i, last_cta);
    }
    pdl_launch_dependents();
    pdl_wait();          // the prepared activation comes from the preceding kernel
    if (tid == 0) {
        mbar_arrive_expect_tx(act_bar, p.act_bytes);
        bulk_g2s(smem_u32(smem + p.off_act), p.act + (blockIdx.x % kActCopies) * p.act_copy_stride, p.act_bytes,
                 act_bar);
        for (uint32_t i = p.pre_issue; i < ring_to; ++i) issue_item(p, smem, i, last_cta);
    }
    bool ok = mbar_wait(act_bar, 0, p.err);

    const uint32_t gi = warp & 3, par = warp >> 2;
    const uint32_t ring = smem_u32(smem + p.off_ring), act_addr = smem_u32(smem + p.off_act);
    const float2 *gs = reinterpret_cast<const float2 *>(smem + p.off_act + p.groups * 256);
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    const uint32_t sw = (uint32_t)(lane & 7);
    for (uint32_t tile = 0; tile < ntile; ++tile) {
        float y0 = 0.f, y1 = 0.f;      // rows lane and lane + 32 of the tile
        for (uint32_t col = par; col < p.nbox; col += 2) {
            const uint32_t item = tile * p.nbox + col, slot = item % p.nslots;
            ok = ok && mbar_wait(bar0 + 8 * slot, (item / p.nslots) & 1, p.err);
            const uint32_t G = col * 4 + gi;
            if (ok && G < p.groups) {
                const uint32_t sa = ring + slot * kItemBytes;
                const uint32_t r0 = sa + lane * 128, r1 = r0 + 4096;
                // group G = 16-byte chunks 2gi, 2gi+1 of the box line, swizzled by row % 8
                const uint32_t ch0 = ((2 * gi) ^ sw) << 4, ch1 = ((2 * gi + 1) ^ sw) << 4;
                const uint4 a0 = lds128u(r0 + ch0), a1 = lds128u(r0 + ch1);
                const uint4 b0 = lds128u(r1 + ch0), b1 = lds128u(r1 + ch1);
                const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                int u0 = 0, u1 = 0, u2 = 0, u3 = 0, v0 = 0, v1 = 0, v2 = 0, v3 = 0;
#pragma unroll
                for (int wi = 0; wi < 8; ++wi) {
                    const uint32_t aw = act_addr + (G * 8 + wi) * 32;
                    const uint4 lo = lds128u(aw), hi = lds128u(aw + 16);
                    const uint32_t ca = wa[wi], cb = wb[wi];
                    u0 = dp2a_hi(hi.x, ca & 0x03030303u, dp2a_lo(lo.x, ca & 0x03030303u, u0));
                    u1 = dp2a_hi(hi.y, ca & 0x0C0C0C0Cu, dp2a_lo(lo.y, ca & 0x0C0C0C0Cu, u1));
                    u2 = dp2a_hi(hi.z, ca & 0x30303030u, dp2a_lo(lo.z, ca & 0x30303030u, u2));
                    u3 = dp2a_hi(hi.w, ca & 0xC0C0C0C0u, dp2a_lo(lo.w, ca & 0xC0C0C0C0u, u3));
                    v0 = dp2a_hi(hi.x, cb & 0x03030303u, dp2a_lo(lo.x, cb & 0x03030303u, v0));
                    v1 = dp2a_hi(hi.y, cb & 0x0C0C0C0Cu, dp2a_lo(lo.y, cb & 0x0C0C0C0Cu, v1));
                    v2 = dp2a_hi(hi.z, cb & 0x30303030u, dp2a_lo(lo.z, cb & 0x30303030u, v2));
                    v3 = dp2a_hi(hi.w, cb & 0xC0C0C0C0u, dp2a_lo(lo.w, cb & 0xC0C0C0C0u, v3));
                }
                const float2 f = gs[G];
                const int off = __float_as_int(f.y);
                const int t0 = u0 + (u1 >> 2) + (u2 >> 4) + (u3 >> 6) - off;
                const int t1 = v0 + (v1 >> 2) + (v2 >> 4) + (v3 >> 6) - off;
                // scale box: row r at r * 16 bytes holds groups 8 * (col / 2) .. + 7
                const uint32_t so = 2 * (4 * (col & 1) + gi);
                const float s0 = __half2float(__ushort_as_half((unsigned short)lds16(sa + 8192 + lane * 16 + so)));
                const float s1 = __half2float(__ushort_as_half((unsigned short)lds16(sa + 8192 + 512 + lane * 16 + so)));
                y0 = fmaf(s0 * f.x, (float)t0, y0);
                y1 = fmaf(s1 * f.x, (float)t1, y1);
            }
            // release the slot; the fourth reader re-arms it with item + nslots
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const uint32_t seen = atomicAdd(&cnt[slot], 1u);
                if (seen == 3) {
                    cnt[slot] = 0;
                    if (ok && item + p.nslots < nitems) {
                        fence_proxy_async();
                        issue_item(p, smem, item + p.nslots, last_cta);
                    }
                }
            }
        }
        part[warp * kRows + lane] = y0;
        part[warp * kRows + 32 + lane] = y1;
        __syncthreads();
        if (warp < 2) {
            const uint32_t rl = warp * 32 + lane;
            const uint64_t r = r_begin + (uint64_t)tile * kRows + rl;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += part[w * kRows + rl];
            if (r < r_end) store1(p.y, r, p.y_dtype, acc);
        }
        __syncthreads();
    }
}

}  // namespace

bool gemv_pq2_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                       IntPlan *plan) {
    *plan = IntPlan{};
    if (M != 1) return false;
    if (rotate && g.k % 1024) return false;
    // scale rows must be whole 16-byte units for the scale boxes
    if (g.scale_row_bytes % 16 || g.base_row_bytes % 16 || g.payload_bytes % 16) return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31)) return false;
    const uint32_t groups = (uint32_t)g.groups_per_row;
    const uint32_t nbox = (uint32_t)((g.base_row_bytes + 127) / 128);
    const uint32_t act_bytes = ((groups * 264 + 15) / 16) * 16;
    const uint32_t part_bytes = kWarps * kRows * 4;
    const uint32_t bar_bytes = (kMaxSlots + 1) * 8;
    const uint32_t fixed = act_bytes + part_bytes + bar_bytes + kMaxSlots * 4;
    // two CTAs per SM share its 228 KB (each CTA also reserves 1 KB)
    const int per_cta = (228 * 1024) / 2 - 1024;
    const int limit = std::min(smem_limit, per_cta);
    if ((int)fixed + 2 * (int)kItemBytes > limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((limit - (int)fixed) / (int)kItemBytes));
    // two CTAs per SM with ~n / (2 * SMs) rows each (tiles of 64 rows, the last
    // one partly out of the CTA's range and never read from HBM)
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>(2ull * (uint64_t)sms, g.n / 32));
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid = (g.n + R - 1) / R;
    plan->ok = true;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nbox = nbox;
    plan->nslots = nslots;
    plan->pre_issue = nslots;      // the whole ring before the dependency wait
    plan->act_bytes = act_bytes;
    plan->off_ring = 0;
    plan->off_act = nslots * kItemBytes;
    plan->off_part = plan->off_act + act_bytes;
    plan->off_bar = plan->off_part + part_bytes;
    plan->off_cnt = plan->off_bar + bar_bytes;
    plan->smem = plan->off_cnt + kMaxSlots * 4;
    plan->workspace = act_prep_int16_row_bytes(g.k_pad) * kActCopies;
    return true;
}

int gemv_pq2_int_launch(const IntPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                        int x_dtype, const uint16_t *signs, void *y, int y_dtype, void *workspace, cudaStream_t stream,
                        bool pdl) {
    int st = act_prep_int16_launch(x, x_dtype, signs, g.k, g.k_pad, 1, kActCopies, static_cast<uint8_t *>(workspace),
                                   stream, pdl);
    if (st) return st;
    IntParams p;
    std::memset(&p, 0, sizeof p);
    const uint8_t *base = payload + g.base_offset, *scale = payload + g.scale_offset;
    p.act = static_cast<const uint8_t *>(workspace);
    p.act_copy_stride = act_prep_int16_row_bytes(g.k_pad);
    p.y = y;
    p.n = g.n;
    p.groups = (uint32_t)g.groups_per_row;
    p.nbox = plan.nbox;
    p.rows_per_cta = plan.rows_per_cta;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.pre_issue = plan.pre_issue;
    p.act_bytes = plan.act_bytes;
    p.off_ring = plan.off_ring;
    p.off_act = plan.off_act;
    p.off_part = plan.off_part;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_cta, G = plan.grid, last_rows = g.n - (G - 1) * R;
    if (G > 1) {
        st = encode_rows(&p.wmap_main, base, g.base_row_bytes, R, G - 1, 128, 32, true);
        if (!st) st = encode_rows(&p.smap_main, scale, g.scale_row_bytes, R, G - 1, 16, 32, false);
        if (st) return st;
    }
    st = encode_rows(&p.wmap_last, base + (G - 1) * R * g.base_row_bytes, g.base_row_bytes, last_rows, 1, 128, 32, true);
    if (!st)
        st = encode_rows(&p.smap_last, scale + (G - 1) * R * g.scale_row_bytes, g.scale_row_bytes, last_rows, 1, 16, 32,
                         false);
    if (st) return st;
    cudaError_t e = cudaFuncSetAttribute(gemv_pq2_int_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv: smem attribute: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_pq2_int_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
