// Decode GEMV for PQ2_0_G128 weights and 2 <= M <= 8 activation rows.
//
// What it computes:
//   y[m][r] = sum_g scale[r][g] * sum_{j<128} (code[r][128g+j] - 1) * xr[m][128g+j]
// with xr the forward-rotated activation (per 1024-block H (D * x) / 32,
// "artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2), codes the
// 2-bit fields of the base plane, least significant first, value = code - 1
// ("GGUF 完整讲解" §4.3), one binary16 scale per 128-weight group
// ("bonsai三元GGUF模型转ninfer模型01" §3).
//
// Arithmetic: mma.sync m16n8k16 with binary16 operands and fp32 accumulators;
// the eight MMA columns are the (up to) eight activation rows.
//  * A (weights): a 32-bit code word holds 16 codes (code j at bits 2j). The
//    mask 0x00030003 << 2c leaves codes c and c + 8 as the binary16 subnormals
//    code * 4^c * 2^-24 (exact); the word shifted right by 8 gives codes c + 4 and
//    c + 12 the same way. Lane c of a quad therefore feeds K slots (c, c + 8,
//    c + 4, c + 12) of every 16-weight word.
//  * B (activations): binary16 of xr * 2^E / 4^c (E per 1024-block and
//    row, so that max |xr * 2^E| < 2^11), written once per call by
//    mma_prep_kernel in the fragment order of the MMA, plus per group and row
//    {2^-E, X} with X the sum of the group's B values times 4^c.
//  * Per group: y += scale * 2^-E * (2^24 * C - X)       (value = code - 1)
// Products of binary16 operands are exact; the sums are fp32.
//
// Data movement: one CTA per SM owns a contiguous row range in tiles of 128
// rows; weights stream through a ring of 34 KB items of 128 rows x 8 groups
// (two 128-byte-swizzled code boxes and one scale box), taken column by column:
// item i covers groups 8j .. 8j + 7 of tile t with j = i / tiles, t = i % tiles.
// Warp w takes the 16-row slice w / 2 and groups 4 (w % 2) .. 4 (w % 2) + 3 of
// every item, so it keeps those four groups' B fragments (64 registers) for a
// whole column of tiles instead of re-reading them from shared memory per tile.
// The fragments arrive per column (16 KB, double-buffered bulk copies from the
// prep kernel's output); the two warps of a slice add their halves through
// shared memory and the sums accumulate per tile in shared memory until the
// last column.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "act16.cuh"
#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
namespace {

constexpr int kThreads = 512;     // 16 warps; one CTA per SM
constexpr int kWarps = 16;
constexpr int kRows = 128;        // rows per tile: 8 slices of 16
constexpr uint32_t kBoxBytes = 128 * kRows;
constexpr uint32_t kItemBytes = 2 * kBoxBytes + 16 * kRows;
constexpr uint32_t kMaxSlots = 8;
constexpr uint32_t kWordFrag = 32 * 8;   // B fragments of one 16-weight word: 32 lanes x 2 registers
constexpr uint32_t kColFrag = 8 * 8 * kWordFrag;   // B fragments of one item column (8 groups)
constexpr uint32_t kTileAcc = 8 * 32 * 16;         // per tile: a float4 per lane of each of the 8 slices
constexpr uint32_t kMaxTiles = 16;                 // tiles per CTA (their sums live in shared memory)

struct MmaParams {
    CUtensorMap wmap_main, wmap_last;   // base rows: {row bytes, R rows, CTA} / last CTA {row bytes, rows}
    CUtensorMap smap_main, smap_last;   // scale rows, same views
    const uint8_t *frag;                // mma_prep_kernel output: fragments, then {2^-E, X} per (group, row)
    uint32_t fx_bytes;
    void *y;
    uint64_t n;
    uint32_t M, groups, nitem, rows_per_cta;
    int y_dtype;
    uint32_t nslots, pre_issue;
    uint32_t off_ring, off_frag, off_fx, off_acc, off_part, off_bar, off_cnt;
    uint32_t *err;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Rotates block b of activation row m and writes its B fragments and group
// entries. Fragment (word W, lane L = 4n + c) of row n = m holds
//   reg 0: (v[16W + c], v[16W + c + 8]),  reg 1: (v[16W + c + 4], v[16W + c + 12])
// with v = binary16(xr * 2^E / 4^c); rows m >= M write zeros.
__global__ void __launch_bounds__(64) mma_prep_kernel(const XSource xsrc, uint64_t row_stride_bytes, uint32_t M,
                                                      uint32_t groups, uint8_t *out) {
    __shared__ __align__(16) float tile[kRotScratch / 4];
    const int t = threadIdx.x, lane = t & 31;
    const uint32_t b = blockIdx.x, m = blockIdx.y;
    const uint32_t words = groups * 8;
    uint16_t *frag = reinterpret_cast<uint16_t *>(out);
    float2 *fx = reinterpret_cast<float2 *>(out + (uint64_t)words * kWordFrag);
    float d[16];
    if (xsrc.signs && m < M) load_signs16(xsrc, b, t, d);     // read-only parameter: before the dependency wait
    pdl_launch_dependents();
    pdl_wait();
    float v[16];
    int E = 0;
    if (m < M) {
        XSource xs = xsrc;
        xs.x = static_cast<const uint8_t *>(xsrc.x) + m * row_stride_bytes;
        load_run16(xs, b, t, v);
        const float mx = rotate16(xsrc.signs != nullptr, t, v, d, tile, 1);
        if (mx > 0.f) E = 10 - ilogbf(mx);      // max |xr * 2^E| < 2^11
        E = max(-100, min(100, E));
    } else {
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = 0.f;
    }
    const float up = ldexpf(1.f, E);
    float gsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        // element 256 (r / 4) + 4t + c, c = r % 4: word 16 (r / 4) + t / 4 of the block, position 4 (t % 4) + c
        const int c = r & 3;
        const __half h = __float2half_rn(v[r] * up * (c == 0 ? 1.f : c == 1 ? 0.25f : c == 2 ? 0.0625f : 0.015625f));
        gsum[r >> 2] += __half2float(h) * (float)(1 << (2 * c));
        const uint32_t W = b * 64 + 16 * (r >> 2) + (t >> 2), j = 4 * (t & 3) + c;
        if (W < words) frag[((uint64_t)W * 32 + 4 * m + c) * 4 + ((j >> 2) & 1) * 2 + (j >> 3)] = __half_as_ushort(h);
    }
    // group of element 256 a + 4t + c: 2a + t / 32 -> reduce over the warp
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        float s = gsum[a];
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) s += __shfl_xor_sync(0xffffffffu, s, sh);
        const uint32_t G = b * 8 + 2 * a + (t >> 5);
        if (lane == 0 && G < groups) fx[G * 8 + m] = make_float2(m < M ? ldexpf(1.f, -E) : 0.f, s);
    }
}

// Item i = j * ntile + t (groups 8j .. 8j + 7 of tile t): its two code boxes
// and its scale box into ring slot i % nslots (one thread).
__device__ __forceinline__ void issue_item(const MmaParams &p, uint8_t *smem, uint32_t item, uint32_t ntile,
                                           bool last_cta) {
    const uint32_t j = item / ntile, tile = item % ntile, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kItemBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kItemBytes);
    const int y0 = (int)(tile * kRows), xs = (int)(j * 16);
    if (last_cta) {
        tma_load_2d(dst, &p.wmap_last, (int)(j * 256), y0, bar);
        tma_load_2d(dst + kBoxBytes, &p.wmap_last, (int)(j * 256 + 128), y0, bar);
        tma_load_2d(dst + 2 * kBoxBytes, &p.smap_last, xs, y0, bar);
    } else {
        tma_load_3d(dst, &p.wmap_main, (int)(j * 256), y0, (int)blockIdx.x, bar);
        tma_load_3d(dst + kBoxBytes, &p.wmap_main, (int)(j * 256 + 128), y0, (int)blockIdx.x, bar);
        tma_load_3d(dst + 2 * kBoxBytes, &p.smap_main, xs, y0, (int)blockIdx.x, bar);
    }
}

// B fragments of item column j (up to 8 groups, 16 KB) into fragment buffer j % 2.
__device__ __forceinline__ void issue_column(const MmaParams &p, uint8_t *smem, uint32_t j, uint32_t bar) {
    const uint32_t ng = p.groups - 8 * j < 8 ? p.groups - 8 * j : 8;
    const uint32_t bytes = ng * 8 * kWordFrag;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(smem + p.off_frag) + (j & 1) * kColFrag, p.frag + (uint64_t)j * kColFrag, bytes, bar);
}

__global__ void __launch_bounds__(kThreads, 1) gemv_pq2_mma_kernel(const __grid_constant__ MmaParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t r_begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t r_end = r_begin + p.rows_per_cta < p.n ? r_begin + p.rows_per_cta : p.n;
    const bool last_cta = blockIdx.x == gridDim.x - 1;
    const uint32_t ntile = (uint32_t)((r_end - r_begin + kRows - 1) / kRows);
    const uint32_t nitems = ntile * p.nitem;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t col_bar = bar0 + 8 * kMaxSlots;      // two: one per fragment buffer
    const uint32_t fx_bar = col_bar + 16;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1, *ccnt = cnt + kMaxSlots + 2;
    uint32_t *col_last = cnt + kMaxSlots + 4;           // last column issued into each fragment buffer

    if (tid == 0) {
        prefetch_tmap(last_cta ? &p.wmap_last : &p.wmap_main);
        prefetch_tmap(last_cta ? &p.smap_last : &p.smap_main);
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        mbar_init(col_bar, 1);
        mbar_init(col_bar + 8, 1);
        mbar_init(fx_bar, 1);
        ccnt[0] = ccnt[1] = 0;
        col_last[0] = 0;
        col_last[1] = p.nitem > 1 ? 1u : 0xffffffffu;
        *failed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    const uint32_t pre = p.pre_issue < ring_to ? p.pre_issue : ring_to;
    if (tid == 0) {
        // weights are read-only parameters: a few items before the dependency wait
        for (uint32_t i = 0; i < pre; ++i) issue_item(p, smem, i, ntile, last_cta);
    }
    pdl_launch_dependents();
    pdl_wait();          // the fragments come from the prep kernel
    if (tid == 0) {
        mbar_arrive_expect_tx(fx_bar, p.fx_bytes);
        bulk_g2s(smem_u32(smem + p.off_fx), p.frag + (uint64_t)p.groups * 8 * kWordFrag, p.fx_bytes, fx_bar);
        issue_column(p, smem, 0, col_bar);
        if (p.nitem > 1) issue_column(p, smem, 1, col_bar + 8);
        for (uint32_t i = pre; i < ring_to; ++i) issue_item(p, smem, i, ntile, last_cta);
        *issued = ring_to;
    }
    bool ok = mbar_wait(fx_bar, 0, p.err);

    const float2 *fx = reinterpret_cast<const float2 *>(smem + p.off_fx);
    float4 *part = reinterpret_cast<float4 *>(smem + p.off_part);
    float4 *acc_s = reinterpret_cast<float4 *>(smem + p.off_acc);
    const uint32_t slice = warp >> 1, gh = warp & 1, g4 = lane >> 2, c = lane & 3;
    const uint32_t mask = 0x00030003u << (2 * c);
    const uint32_t r0 = slice * 16 + g4, r1 = r0 + 8;     // tile rows of this lane (MMA rows g4, g4 + 8)
    const bool refill = nitems > p.nslots;
    uint2 bfr[4][8];
    uint32_t slot = 0, phase = 0, tile = 0, j = 0;
    for (uint32_t it = 0; it < nitems; ++it) {
        if (tile == 0) {
            // this warp's B fragments of column j; the last of the sixteen warps to
            // take them refills the buffer with column j + 2
            ok = ok && mbar_wait(col_bar + 8 * (j & 1), (j >> 1) & 1, p.err);
            const uint2 *fw = reinterpret_cast<const uint2 *>(smem + p.off_frag + (j & 1) * kColFrag) + lane;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int w = 0; w < 8; ++w) bfr[q][w] = fw[((4 * gh + q) * 8 + w) * 32];
            __syncwarp();
            if (lane == 0) {
                if (!ok) *failed = 1;
                __threadfence_block();
                const uint32_t seen = atomicAdd(&ccnt[j & 1], 1u);
                if (seen == kWarps - 1) {
                    ccnt[j & 1] = 0;
                    if (ok && !*(volatile uint32_t *)failed && j + 2 < p.nitem) {
                        fence_proxy_async();
                        issue_column(p, smem, j + 2, col_bar + 8 * (j & 1));
                        col_last[j & 1] = j + 2;
                    }
                }
            }
            __syncwarp();
        }
        ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err);
        float a4[4] = {0.f, 0.f, 0.f, 0.f};       // rows r0, r1 x activation rows 2c, 2c + 1
        if (ok) {
            const uint8_t *sa = smem + p.off_ring + slot * kItemBytes;
            const uint8_t *bx = sa + gh * kBoxBytes;     // groups 4 gh .. 4 gh + 3 = box gh
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t gl = 4 * gh + q, G = j * 8 + gl;
                if (G < p.groups) {
                    // group gl = 16-byte chunks 2q, 2q + 1 of its box, swizzled by row % 8
                    float C[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(bx + r0 * 128 + (((2 * q + hf) ^ (r0 & 7)) << 4));
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(bx + r1 * 128 + (((2 * q + hf) ^ (r1 & 7)) << 4));
                        const uint32_t cw0[4] = {w0.x, w0.y, w0.z, w0.w}, cw1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const uint2 bf = bfr[q][4 * hf + qq];
                            mma16816(C, cw0[qq] & mask, cw1[qq] & mask, (cw0[qq] >> 8) & mask, (cw1[qq] >> 8) & mask,
                                     bf.x, bf.y);
                        }
                    }
                    // scale box: row r at r * 16 bytes holds the item's 8 scales
                    const float s0 = __half2float(*reinterpret_cast<const __half *>(sa + 2 * kBoxBytes + r0 * 16 + 2 * gl));
                    const float s1 = __half2float(*reinterpret_cast<const __half *>(sa + 2 * kBoxBytes + r1 * 16 + 2 * gl));
                    const float2 f0 = fx[G * 8 + 2 * c], f1 = fx[G * 8 + 2 * c + 1];
                    a4[0] = fmaf(s0 * f0.x, fmaf(C[0], 16777216.f, -f0.y), a4[0]);
                    a4[1] = fmaf(s0 * f1.x, fmaf(C[1], 16777216.f, -f1.y), a4[1]);
                    a4[2] = fmaf(s1 * f0.x, fmaf(C[2], 16777216.f, -f0.y), a4[2]);
                    a4[3] = fmaf(s1 * f1.x, fmaf(C[3], 16777216.f, -f1.y), a4[3]);
                }
            }
        }
        if (refill) {
            // release the slot; the last of the sixteen readers re-arms it with item + nslots
            __syncwarp();
            if (lane == 0) {
                if (!ok) *failed = 1;
                __threadfence_block();
                const uint32_t seen = atomicAdd(&cnt[slot], 1u);
                if (seen == kWarps - 1) {
                    cnt[slot] = 0;
                    if (ok && !*(volatile uint32_t *)failed && it + p.nslots < nitems) {
                        fence_proxy_async();
                        issue_item(p, smem, it + p.nslots, ntile, last_cta);
                        atomicAdd(issued, 1u);
                    }
                }
            }
            __syncwarp();
        } else if (!ok && lane == 0) {
            *failed = 1;
        }
        if (++slot == p.nslots) {
            slot = 0;
            phase ^= 1u;
        }
        // the two warps of a slice hold complementary group halves: the even warp
        // adds them into the tile's sums
        float4 *pb = part + ((it & 1) * 8 + slice) * 32 + lane;
        if (gh) *pb = make_float4(a4[0], a4[1], a4[2], a4[3]);
        named_barrier(1 + slice, 64);
        if (!gh) {
            const float4 o = *pb;
            float4 *as = acc_s + (tile * 8 + slice) * 32 + lane;
            float4 v = make_float4(a4[0] + o.x, a4[1] + o.y, a4[2] + o.z, a4[3] + o.w);
            if (j) {
                const float4 prev = *as;
                v = make_float4(prev.x + v.x, prev.y + v.y, prev.z + v.z, prev.w + v.w);
            }
            *as = v;
        }
        if (++tile == ntile) {
            tile = 0;
            ++j;
        }
    }
    if (!gh) {
        // this warp's rows of every tile, activation rows 2c and 2c + 1
        for (uint32_t t = 0; t < ntile; ++t) {
            const float4 v = acc_s[(t * 8 + slice) * 32 + lane];
            const float sum[4] = {v.x, v.y, v.z, v.w};
            const uint64_t row[2] = {r_begin + (uint64_t)t * kRows + r0, r_begin + (uint64_t)t * kRows + r1};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint64_t r = row[i >> 1];
                const uint32_t m = 2 * c + (i & 1);
                if (r < r_end && m < p.M) store1(p.y, (uint64_t)m * p.n + r, p.y_dtype, sum[i]);
            }
        }
    }
    // after a timed-out wait: let the copies still in flight land (at most one
    // per slot, the last one issued into it) before the CTA's memory is freed
    __syncthreads();
    if (tid == 0 && *(volatile uint32_t *)failed) {
        const uint32_t n_issued = *(volatile uint32_t *)issued;
        for (uint32_t i = n_issued > p.nslots ? n_issued - p.nslots : 0; i < n_issued; ++i)
            mbar_wait(bar0 + 8 * (i % p.nslots), (i / p.nslots) & 1, p.err, 200000000ll);
        mbar_wait(fx_bar, 0, p.err, 200000000ll);
        for (uint32_t b = 0; b < 2; ++b) {
            const uint32_t jl = *(volatile uint32_t *)&col_last[b];
            if (jl != 0xffffffffu) mbar_wait(col_bar + 8 * b, (jl >> 1) & 1, p.err, 200000000ll);
        }
    }
}

}  // namespace

bool gemv_pq2_mma_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                       MmaPlan *plan) {
    *plan = MmaPlan{};
    if (M < 2 || M > 8) return false;
    if (rotate && g.k % 1024) return false;
    if (g.k % 8) return false;     // rows of x after the first stay 16-byte aligned for the vector loads
    if (g.scale_row_bytes % 16 || g.base_row_bytes % 16 || g.payload_bytes % 16) return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31)) return false;
    const uint32_t groups = (uint32_t)g.groups_per_row;
    // one CTA per SM with ~n / SMs rows each, at most kMaxTiles tiles of sums per CTA
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)sms, g.n / 64));
    uint64_t R = (g.n + grid0 - 1) / grid0;
    R = std::min<uint64_t>(R, (uint64_t)kMaxTiles * kRows);
    const uint64_t grid = (g.n + R - 1) / R;
    const uint32_t ntile = (uint32_t)((R + kRows - 1) / kRows);
    const uint32_t fx_bytes = groups * 8 * 8;
    const uint32_t acc_bytes = ntile * kTileAcc;
    const uint32_t part_bytes = 2 * 8 * 32 * 16;
    const uint32_t bar_bytes = (kMaxSlots + 3) * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 8) * 4;
    const uint32_t fixed = 2 * kColFrag + fx_bytes + acc_bytes + part_bytes + bar_bytes + cnt_bytes;
    if ((int64_t)fixed + 2 * (int64_t)kItemBytes > smem_limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((smem_limit - (int)fixed) / (int)kItemBytes));
    plan->ok = true;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nitem = (groups + 7) / 8;
    plan->nslots = nslots;
    plan->pre_issue = std::min<uint32_t>(1, nslots);
    plan->fx_bytes = fx_bytes;
    uint32_t off = 0;
    plan->off_ring = off;
    off += nslots * kItemBytes;
    plan->off_frag = off;
    off += 2 * kColFrag;
    plan->off_fx = off;
    off += fx_bytes;
    plan->off_acc = off;
    off += acc_bytes;
    plan->off_part = off;
    off += part_bytes;
    plan->off_bar = off;
    off += bar_bytes;
    plan->off_cnt = off;
    off += cnt_bytes;
    plan->smem = off;
    plan->workspace = (uint64_t)groups * 8 * kWordFrag + fx_bytes;
    return true;
}

int gemv_pq2_mma_launch(const MmaPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                        int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, void *workspace,
                        cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    {
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3((unsigned)((g.k + 1023) / 1024), 8);
        pc.blockDim = dim3(64);
        pc.stream = stream;
        pc.attrs = attr;
        pc.numAttrs = 1;
        const XSource xsrc{x, signs, (uint32_t)g.k, x_dtype};
        cudaError_t e = cudaLaunchKernelEx(&pc, mma_prep_kernel, xsrc, (uint64_t)(g.k * dtype_size(x_dtype)),
                                           (uint32_t)M, (uint32_t)g.groups_per_row, static_cast<uint8_t *>(workspace));
        if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "decode prep launch: %s", cudaGetErrorString(e));
    }
    MmaParams p;
    std::memset(&p, 0, sizeof p);
    const uint8_t *base = payload + g.base_offset, *scale = payload + g.scale_offset;
    p.frag = static_cast<const uint8_t *>(workspace);
    p.fx_bytes = plan.fx_bytes;
    p.y = y;
    p.n = g.n;
    p.M = (uint32_t)M;
    p.groups = (uint32_t)g.groups_per_row;
    p.nitem = plan.nitem;
    p.rows_per_cta = plan.rows_per_cta;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.pre_issue = plan.pre_issue;
    p.off_ring = plan.off_ring;
    p.off_frag = plan.off_frag;
    p.off_fx = plan.off_fx;
    p.off_acc = plan.off_acc;
    p.off_part = plan.off_part;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_cta, G = plan.grid, last_rows = g.n - (G - 1) * R;
    if (G > 1) {
        st = encode_row_tiles(&p.wmap_main, base, g.base_row_bytes, R, G - 1, 128, kRows, true);
        if (!st) st = encode_row_tiles(&p.smap_main, scale, g.scale_row_bytes, R, G - 1, 16, kRows, false);
        if (st) return st;
    }
    st = encode_rows(&p.wmap_last, base + (G - 1) * R * g.base_row_bytes, g.base_row_bytes, last_rows, 128, kRows,
                     true);
    if (!st)
        st = encode_rows(&p.smap_last, scale + (G - 1) * R * g.scale_row_bytes, g.scale_row_bytes, last_rows, 16,
                         kRows, false);
    if (st) return st;
    int st_attr = set_smem_attribute((const void *)gemv_pq2_mma_kernel, (int)plan.smem);
    if (st_attr) return st_attr;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_pq2_mma_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "decode gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
