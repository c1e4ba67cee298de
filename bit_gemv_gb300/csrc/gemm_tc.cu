// Prefill projection for PQ2_0_G128 (M > 8 activation rows) on the 5th-generation
// tensor cores: tcgen05.mma kind::f16, fp32 accumulators in tensor memory.
//
// What it computes:
//   y[m][r] = sum_c W[r][c] * xr[m][c],  W[r][c] = (code[r][c] - 1) * scale[r][c / 128]
// with xr the forward-rotated activation (per 1024-block H (D * x) / 32,
// "artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2), codes the
// 2-bit fields of the base plane, least significant first, value = code - 1
// ("GGUF 完整讲解" §4.3), one binary16 scale per 128-weight group
// ("bonsai三元GGUF模型转ninfer模型01" §3).
//
// Precision: xr is rounded to binary16 once; W = (code - 1) * scale is exact in
// binary16 (a small integer times a binary16 value); products are exact and
// accumulate in fp32.
//
// Two kernels:
//  * tc_prep_kernel writes xr as binary16, one warp per (row, 1024-block). Inside
//    every run of 16 elements it stores the order 0,8,1,9,...,7,15, which is the
//    order in which one 32-bit word of codes decodes with one mask per pair
//    (codes j and j+8 sit at bits 2j and 2j+16).
//  * gemm_tc_kernel is persistent: one CTA per SM walks the output tiles
//    (128 weight rows x 192 tokens) t = blockIdx.x, blockIdx.x + gridDim.x, ...,
//    K in stages of 64. The expanded weights are the MMA's A operand and live in
//    tensor memory, so they never pass through shared memory; xr is the B
//    operand, in shared memory. Two accumulator buffers in tensor memory let the
//    epilogue of one tile run under the main loop of the next:
//      warp 0       TMA producer: xr tile (192 tokens x 64 binary16, 128-byte
//                   swizzle), the tile's 64 codes per weight row (16 bytes) and
//                   the 8 scales that cover them (16 bytes);
//      warp 1       TMEM owner and MMA issuer (one thread): four K=16 MMAs per
//                   stage into the tile's accumulator buffer;
//      warps 2..9   decode: lane l of warp w expands weight row 32 (w % 4) + l
//                   (its tensor-memory lane) to binary16 (code - 1) * scale and
//                   stores 16 of the stage's 32 binary16 pairs into the stage's
//                   A columns (warps 2..5 the first 16, warps 6..9 the rest);
//      warps 10..13 epilogue: read a finished accumulator buffer (lane = weight
//                   row, column = token), store y, hand the buffer back.
//    Stages and buffers are handed over with mbarriers (TMA transaction counts,
//    one arrival per decode or epilogue warp, and tcgen05.commit for "stage
//    consumed" and "tile accumulated"); every wait is bounded.
#include <algorithm>
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
namespace {

constexpr int kBM = 192, kBN = 128, kBK = 64;      // tokens (MMA N), weight rows (MMA M), k per stage
constexpr int kStages = 4;
constexpr uint32_t kXBytes = kBM * kBK * 2;        // 24 KB of xr
constexpr uint32_t kCodeBytes = kBN * 16;          // 64 codes per weight row
constexpr uint32_t kScaleBytes = kBN * 16;         // 8 scales per weight row
constexpr uint32_t kStageBytes = kXBytes + kCodeBytes + kScaleBytes;     // 28 KB, 1024-aligned
constexpr uint32_t kBarBytes = 8 * (3 * kStages + 4);
constexpr uint32_t kSmemBytes = ((kStages * kStageBytes + kBarBytes + 16 + 1023) / 1024) * 1024;
constexpr int kThreads = 448;
constexpr uint32_t kAccCols = kBM;                 // one fp32 accumulator buffer: lane = weight row, column = token
constexpr uint32_t kACols = kBK / 2;               // a stage's weights per row, as binary16 pairs
constexpr uint32_t kAColBase = 2 * kAccCols;       // A stages after the two accumulator buffers
constexpr uint32_t kTmemCols = 512;                // a power of two; one CTA per SM
static_assert(kAColBase + kStages * kACols <= kTmemCols, "tensor memory plan");
static_assert(kStageBytes % 1024 == 0, "swizzled xr tiles need 1024-byte alignment");

struct TcParams {
    CUtensorMap amap, cmap, smap;
    void *y;
    uint64_t M, n;
    uint32_t nk, gn, tiles;     // K stages, weight tiles, tiles (weight tile fastest)
    int y_dtype;
    uint32_t *err;
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (8-row atoms of
// 1024 bytes), start address in 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 D, binary16 A and B, both K-major,
// M = 128 (weight rows), N = 192 (tokens).
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kBM >> 3) << 17) | ((uint32_t)(kBN >> 4) << 24);

// D (tensor memory) += A (tensor memory, M x 16) * B (shared memory descriptor, 16 x N).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes, from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Codes j and j+8 of a 32-bit code word as a binary16 pair ((c - 1) * s):
// OR-ing 0x6400 (1024.0) over a 2-bit code gives 1024 + c exactly.
__device__ __forceinline__ uint32_t expand_pair(uint32_t w, int j, __half2 s2) {
    uint32_t u = ((w >> (2 * j)) & 0x00030003u) | 0x64006400u;
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    h = __hmul2(__hsub2(h, __float2half2_rn(1025.f)), s2);
    return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(128) tc_prep_kernel(const void *__restrict__ x, int x_dtype,
                                                      const uint16_t *__restrict__ signs, __half *__restrict__ out,
                                                      uint64_t M, uint64_t K) {
    // per warp: its 1024-block, element e at e + 8 (e >> 8) (padding keeps the
    // transposed reads conflict-free)
    __shared__ __align__(16) float tile_s[4][1024 + 32];
    const uint64_t nblk = K / 1024;
    const uint64_t task = (uint64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (task >= M * nblk) return;
    const int lane = threadIdx.x & 31;
    float *t = tile_s[threadIdx.x >> 5];
    const uint64_t m = task / nblk, b = task % nblk;
    const uint64_t row = m * K, col0 = b * 1024;
    // lane l holds v[8 i + e] = element 256 i + 8 l + e: index bits 0-2 and 8-9 in registers
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float tv[8];
        const uint64_t c = col0 + 256 * i + 8 * lane;
        load8(x, row + c, x_dtype, tv);
        if (signs) {
            float d[8];
            load_signs8(signs, c, d);
#pragma unroll
            for (int e = 0; e < 8; ++e) tv[e] *= d[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * i + e] = tv[e];
    }
    if (signs) {
#pragma unroll
        for (int bit = 0; bit < 5; ++bit)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j & (1 << bit)) continue;
                const float a = v[j], c = v[j | (1 << bit)];
                v[j] = a + c;
                v[j | (1 << bit)] = a - c;
            }
    }
    // transpose through shared memory: lane l' = (i', e') = (l' >> 3, l' & 7)
    // then holds w[r] = element 256 i' + 8 r + e', index bits 3-7 in registers
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 *dst = reinterpret_cast<float4 *>(t + 264 * i + 8 * lane);
        dst[0] = make_float4(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3]);
        dst[1] = make_float4(v[8 * i + 4], v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]);
    }
    __syncwarp();
    const int ip = lane >> 3, ep = lane & 7;
    float w[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = t[264 * ip + 8 * r + ep];
    if (signs) {
#pragma unroll
        for (int bit = 0; bit < 5; ++bit)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j & (1 << bit)) continue;
                const float a = w[j], c = w[j | (1 << bit)];
                w[j] = a + c;
                w[j | (1 << bit)] = a - c;
            }
#pragma unroll
        for (int r = 0; r < 32; ++r) w[r] *= 0.03125f;
    }
    // output order inside every run of 16: 0,8,1,9,...,7,15. The pair at
    // positions 2e', 2e' + 1 of run 16 s + 256 i' is (w[2 s], w[2 s + 1]).
    uint32_t *o = reinterpret_cast<uint32_t *>(out + row + col0 + 256 * ip + 2 * ep);
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        __half2 p2 = __floats2half2_rn(w[2 * s], w[2 * s + 1]);
        o[8 * s] = *reinterpret_cast<uint32_t *>(&p2);
    }
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(smem);
    if (base & 1023) {         // the swizzled tiles need 1024-byte alignment: report, touch nothing
        if (tid == 0) atomicOr(p.err, kErrSmemAlign);
        return;
    }
    const uint32_t bar = base + kStages * kStageBytes;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kStages * kStageBytes + kBarBytes);
    // full_a[s]: xr, codes and scales landed; full_b[s]: weights expanded into the
    // stage's A columns; empty[s]: stage consumed (shared memory and A columns);
    // acc_full[b]: buffer b holds a finished tile; acc_empty[b]: buffer b read out
#define FULL_A(s) (bar + 8 * (s))
#define FULL_B(s) (bar + 8 * (kStages + (s)))
#define EMPTY(s) (bar + 8 * (2 * kStages + (s)))
#define ACC_FULL(b) (bar + 8 * (3 * kStages + (b)))
#define ACC_EMPTY(b) (bar + 8 * (3 * kStages + 2 + (b)))

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        prefetch_tmap(&p.amap);
        prefetch_tmap(&p.cmap);
        prefetch_tmap(&p.smap);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(FULL_A(s), 1);
            mbar_init(FULL_B(s), 8);
            mbar_init(EMPTY(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(ACC_FULL(b), 1);
            mbar_init(ACC_EMPTY(b), 4);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = 0;     // stage counter over all of this CTA's tiles
            bool ok = true;
            for (uint32_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                const int n0 = (int)((tile % p.gn) * kBN), m0 = (int)((tile / p.gn) * kBM);
                for (uint32_t kt = 0; kt < p.nk; ++kt, ++g) {
                    const uint32_t s = g % kStages, round = g / kStages;
                    if (round > 0 && !mbar_wait(EMPTY(s), (round - 1) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + s * kStageBytes;
                    mbar_arrive_expect_tx(FULL_A(s), kXBytes + kCodeBytes + kScaleBytes);
                    tma_load_2d(st, &p.amap, (int)(kt * kBK), m0, FULL_A(s));
                    tma_load_2d(st + kXBytes, &p.cmap, (int)(kt * 16), n0, FULL_A(s));
                    tma_load_2d(st + kXBytes + kCodeBytes, &p.smap, (int)((kt / 16) * 16), n0, FULL_A(s));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = 0, j = 0;
            bool ok = true;
            for (uint32_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x, ++j) {
                const uint32_t b = j & 1;
                // the buffer's previous tile (two tiles back) has been read out
                if (j >= 2 && !mbar_wait(ACC_EMPTY(b), ((j >> 1) - 1) & 1, p.err)) break;
                tc_fence_after();
                const uint32_t dcol = tmem + b * kAccCols;
                for (uint32_t kt = 0; kt < p.nk; ++kt, ++g) {
                    const uint32_t s = g % kStages, par = (g / kStages) & 1;
                    if (!mbar_wait(FULL_A(s), par, p.err) || !mbar_wait(FULL_B(s), par, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = sw128_desc(base + s * kStageBytes);
                    const uint32_t acol = tmem + kAColBase + kACols * s;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)      // A: +8 columns, B: +32 bytes (16-byte units: +2) per K=16
                        mma_f16_tmem_a(dcol, acol + 8 * kk, bdesc + 2 * kk, (kt | kk) != 0);
                    mma_commit(EMPTY(s));
                }
                if (ok) mma_commit(ACC_FULL(b));
            }
        }
    } else if (warp < 10) {
        // warp w may touch TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31: its lane l is weight row 32 (w % 4) + l;
        // warps 2..5 expand code words 0, 1 of every stage, warps 6..9 words 2, 3
        const uint32_t q = warp & 3, hf = (warp - 2) >> 2;
        const uint32_t r = 32 * q + lane;
        const uint32_t lane_addr = tmem + ((32u * q) << 16);
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
            for (uint32_t kt = 0; kt < p.nk; ++kt, ++g) {
                const uint32_t s = g % kStages, par = (g / kStages) & 1;
                // warp-uniform: the tensor-memory store below is a warp-wide instruction
                if (!__all_sync(0xffffffffu, mbar_wait(FULL_A(s), par, p.err))) {
                    ok = false;
                    break;
                }
                const uint8_t *st = smem + s * kStageBytes;
                const uint4 cw = *reinterpret_cast<const uint4 *>(st + kXBytes + r * 16);
                const __half sc =
                    *reinterpret_cast<const __half *>(st + kXBytes + kCodeBytes + r * 16 + 2 * ((kt / 2) % 8));
                const __half2 s2 = __halves2half2(sc, sc);
                const uint32_t w[2] = {hf ? cw.z : cw.x, hf ? cw.w : cw.y};
                // column 8 i + j holds the pair (code 16 i + j, code 16 i + j + 8): the
                // K order 0,8,1,9,... of every run of 16, as xr is stored
                uint32_t a[16];
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) a[8 * i + jj] = expand_pair(w[i], jj, s2);
                tmem_st16(lane_addr + kAColBase + kACols * s + 16 * hf, a);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(FULL_B(s));
            }
        }
    } else {
        // epilogue: lane = weight row n0 + r of the tile, columns = its tokens
        const uint32_t q = warp & 3;
        const uint32_t r = 32 * q + lane;
        const uint32_t lane_addr = tmem + ((32u * q) << 16);
        uint32_t j = 0;
        for (uint32_t tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++j) {
            const uint32_t b = j & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(ACC_FULL(b), (j >> 1) & 1, p.err))) break;
            tc_fence_after();
            const uint64_t row = (uint64_t)(tile % p.gn) * kBN + r, m0 = (uint64_t)(tile / p.gn) * kBM;
#pragma unroll 1
            for (int cb = 0; cb < kBM / 32; ++cb) {
                float v[32];
                tmem_ld32(lane_addr + b * kAccCols + 32 * cb, v);
                const uint64_t mb = m0 + 32 * cb;
                if (row >= p.n || mb >= p.M) continue;
                const int cnt = p.M - mb < 32 ? (int)(p.M - mb) : 32;
                if (p.y_dtype == NINFER_F32) {
                    float *yp = static_cast<float *>(p.y) + mb * p.n + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < cnt) yp[(uint64_t)i * p.n] = v[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < cnt) store1(p.y, (mb + i) * p.n + row, p.y_dtype, v[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ACC_EMPTY(b));
        }
    }
#undef FULL_A
#undef FULL_B
#undef EMPTY
#undef ACC_FULL
#undef ACC_EMPTY
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

bool gemm_tc_plan(const ninfer_row_split_geometry &g, uint64_t M, int sms, int smem_limit, TcPlan *plan) {
    *plan = TcPlan{};
    if (M < 9 || g.k % 1024 || g.k > (1u << 24)) return false;
    if (g.scale_row_bytes % 16 || g.base_row_bytes % 16) return false;
    if (120 * 1024 > smem_limit || (int)kSmemBytes > smem_limit) return false;
    const uint64_t gm = (M + kBM - 1) / kBM, gn = (g.n + kBN - 1) / kBN;
    if (sms < 1 || gm * gn > 0x7fffffffull || g.n > 0x7fffffffull || M > 0x7fffffffull) return false;
    plan->ok = true;
    plan->grid_n = (uint32_t)gn;
    plan->grid_m = (uint32_t)gm;
    plan->grid = (uint32_t)std::min<uint64_t>((uint64_t)sms, gm * gn);     // persistent: one CTA per SM
    // more than half of an SM's shared memory, so that the persistent CTAs never share an SM
    // (each holds all 512 tensor-memory columns)
    plan->smem = std::max<uint32_t>(kSmemBytes, 120 * 1024);
    plan->workspace = M * g.k * 2;      // xr, binary16
    return true;
}

int gemm_tc_launch(const TcPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                   int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, void *workspace,
                   cudaStream_t stream) {
    __half *xr = static_cast<__half *>(workspace);
    const uint64_t tasks = M * (g.k / 1024), pgrid = (tasks + 3) / 4;
    if (pgrid > 0x7fffffffull) return fail(NINFER_ERR_SHAPE, "prefill: too many rows");
    tc_prep_kernel<<<(unsigned)pgrid, 128, 0, stream>>>(x, x_dtype, signs, xr, M, g.k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "prefill prep launch: %s", cudaGetErrorString(e));
    TcParams p;
    std::memset(&p, 0, sizeof p);
    p.y = y;
    p.M = M;
    p.n = g.n;
    p.nk = (uint32_t)(g.k / kBK);
    p.gn = plan.grid_n;
    p.tiles = plan.grid_n * plan.grid_m;
    p.y_dtype = y_dtype;
    int st = device_error_word(&p.err);
    if (st) return st;
    st = encode_2d(&p.amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xr, g.k, M, g.k * 2, kBK, kBM, true);
    if (!st) st = encode_rows(&p.cmap, payload + g.base_offset, g.base_row_bytes, g.n, 16, kBN, false);
    if (!st) st = encode_rows(&p.smap, payload + g.scale_offset, g.scale_row_bytes, g.n, 16, kBN, false);
    if (st) return st;
    int st_attr = set_smem_attribute((const void *)gemm_tc_kernel, (int)plan.smem);
    if (st_attr) return st_attr;
    gemm_tc_kernel<<<plan.grid, kThreads, plan.smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
