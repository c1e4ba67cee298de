// Decode GEMV for PQ2_0_G128 weights and one activation row (M = 1), on the
// CUDA cores' integer pipes, with the activation rotation fused in.
//
// What it computes:
//   y[r] = sum_g scale[r][g] * sum_{j<128} (code[r][128g+j] - 1) * xr[128g+j]
// with xr the forward-rotated activation, per 1024-block H (D * x) / 32
// ("artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2), codes
// the 2-bit fields of the base plane, least significant first, value = code - 1
// ("GGUF 完整讲解" §4.3), and one binary16 scale per 128-weight group at
// scale_offset ("bonsai三元GGUF模型转ninfer模型01" §3).
//
// Arithmetic: every CTA rotates x itself (one warp per 1024-block: sign
// multiply, the 1024-point butterfly, block maximum) and keeps it in shared
// memory as 16-bit fixed point, x16 = rint(xr * 2^E) with E per block so that
// max |x16| < 2^14, laid out as dp2a operands. In a 32-bit word of codes (16
// weights, four per byte) the mask 0x03 << 2p per byte leaves the four codes of
// position p as bytes (times 4^p); dp2a multiplies two of them by two int16
// activations and accumulates exactly in int32. Per group:
//   sum_j c_j x16_j = acc0 + acc1/4 + acc2/16 + acc3/64        (exact shifts)
//   y += scale * 2^-E * (that - sum_j x16_j)                     (value = code - 1)
// dp2a issues on the FMA-heavy pipe and the masks on the ALU pipe, so the two
// overlap; legacy mma.sync with changing operands is slower on GB300.
//
// Data movement: one CTA per SM owns a contiguous row range, in tiles of 128
// rows. Weights stream through a ring of item slots; an item is 128 rows x 8
// groups: two 128-byte-swizzled tensor boxes of 128 rows x 128 bytes (a 3-D
// map view keeps them inside the CTA's rows) and one box of the rows' 8 scales
// (128 rows x 16 bytes), completing on the slot's mbarrier. Warps w and w + 8
// take words 0-3 and 4-7 of group w of every item, lane l rows l, l+32, l+64,
// l+96 of the tile, so each activation word read from shared memory serves
// four rows. A few items are
// requested before the programmatic-dependent-launch wait (weights and signs
// are read-only parameters, so the stream overlaps the previous kernel's
// tail); x is requested right after the wait and the rest of the ring behind
// it, so the latency-critical read does not queue behind the whole slice. The
// last of the sixteen warps reading an item re-arms its slot with the item
// nslots further on.
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "act16.cuh"
#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {
namespace {

constexpr int kThreads = 512;     // 16 warps, two per group of an item; one CTA per SM
constexpr int kWarps = 16;
constexpr int kRows = 128;        // rows per tile, four per lane
constexpr uint32_t kBoxBytes = 128 * kRows;              // one 128-byte column of the tile
constexpr uint32_t kItemBytes = 2 * kBoxBytes + 16 * kRows;
constexpr uint32_t kMaxSlots = 8;
constexpr uint32_t kRotPairs = 8;     // warp pairs that rotate x (one 1024-block at a time each)

struct IntParams {
    CUtensorMap wmap_main, wmap_last;   // base rows: {row bytes, R rows, CTA} / last CTA {row bytes, rows}
    CUtensorMap smap_main, smap_last;   // scale rows, same views
    CUtensorMap wmap2_main, wmap2_last, smap2_main, smap2_last;     // second matrix (fused gate/up: up)
    const void *x;
    const uint16_t *signs;              // bf16 +-1 per element, or null (no rotation)
    const uint16_t *signs2;             // second matrix's signs (may equal signs)
    uint32_t act_bytes;                 // operand words + group entries of one rotation
    void *y;
    uint64_t n;
    uint32_t k, groups, nblk, nitem, rows_per_cta;     // nitem: items per tile, ceil(groups / 8)
    int x_dtype, y_dtype;
    uint32_t nslots, pre_issue;
    uint32_t off_ring, off_act, off_part, off_bar, off_cnt;
    uint32_t *err;
};

// Item i = tile * (kMats * nitem) + mat * nitem + j (groups 8j .. 8j + 7 of
// the tile's rows of matrix mat): its two weight boxes and its scale box into
// ring slot i % nslots (one thread).
template <int kMats>
__device__ __forceinline__ void issue_item(const IntParams &p, uint8_t *smem, uint32_t item, bool last_cta) {
    const uint32_t per_tile = kMats * p.nitem;
    const uint32_t tile = item / per_tile, jj = item % per_tile, mat = kMats == 1 ? 0 : jj / p.nitem;
    const uint32_t j = jj - mat * p.nitem, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kItemBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kItemBytes);
    const int y0 = (int)(tile * kRows), xs = (int)(j * 16);
    if (last_cta) {
        const CUtensorMap *wm = mat ? &p.wmap2_last : &p.wmap_last, *sm = mat ? &p.smap2_last : &p.smap_last;
        tma_load_2d(dst, wm, (int)(j * 256), y0, bar);
        tma_load_2d(dst + kBoxBytes, wm, (int)(j * 256 + 128), y0, bar);
        tma_load_2d(dst + 2 * kBoxBytes, sm, xs, y0, bar);
    } else {
        const CUtensorMap *wm = mat ? &p.wmap2_main : &p.wmap_main, *sm = mat ? &p.smap2_main : &p.smap_main;
        tma_load_3d(dst, wm, (int)(j * 256), y0, (int)blockIdx.x, bar);
        tma_load_3d(dst + kBoxBytes, wm, (int)(j * 256 + 128), y0, (int)blockIdx.x, bar);
        tma_load_3d(dst + 2 * kBoxBytes, sm, xs, y0, (int)blockIdx.x, bar);
    }
}

// Writes block b's dp2a operand words and group entries (x16 from
// rotate_quantize16, act16.cuh):
//   act[word][4h + p] = (x16[16 word + 8h + p], x16[16 word + 8h + 4 + p]),
//   gs[group] = {2^-E, sum of the group's x16 (as int bits)}.
// Thread t of the pair takes runs t and t + 64 of eight consecutive elements.
__device__ __forceinline__ void pack_pq2(const int16_t *qs, uint8_t *act_s, uint32_t groups, uint32_t b, int t, int E,
                                         uint32_t bar) {
    const int lane = t & 31;
    uint4 *act = reinterpret_cast<uint4 *>(act_s);
    float2 *gs = reinterpret_cast<float2 *>(act_s + (uint64_t)groups * 256);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int run = t + 64 * i;
        const uint4 raw = reinterpret_cast<const uint4 *>(qs)[run];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};     // x16 pairs (2e, 2e+1)
        // entry p = (x16[p], x16[4 + p]) of the run
        uint4 pk;
        pk.x = __byte_perm(w[0], w[2], 0x5410);
        pk.y = __byte_perm(w[0], w[2], 0x7632);
        pk.z = __byte_perm(w[1], w[3], 0x5410);
        pk.w = __byte_perm(w[1], w[3], 0x7632);
        const uint32_t word = b * 64 + (run >> 1);
        if (word < groups * 8) act[word * 2 + (run & 1)] = pk;
        int sum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) sum += (int)(int16_t)(w[q] & 0xffff) + (int)(int16_t)(w[q] >> 16);
#pragma unroll
        for (int sh = 8; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
        const uint32_t G = b * 8 + (run >> 4);     // 16 runs per group of 128
        if ((lane & 15) == 0 && G < groups) gs[G] = make_float2(ldexpf(1.f, -E), __int_as_float(sum));
    }
    named_barrier(bar, 64);      // qs is read before the next block reuses the tile
}

// kMats = 1: y = W x. kMats = 2 (fused FFN gate/up): y = silu(Wg x_g) * (Wu x_u)
// for the same rows of both matrices, x_g and x_u rotated with each matrix's signs.
template <int kMats>
__global__ void __launch_bounds__(kThreads, 1) gemv_pq2_int_kernel(const __grid_constant__ IntParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t r_begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t r_end = r_begin + p.rows_per_cta < p.n ? r_begin + p.rows_per_cta : p.n;
    const bool last_cta = blockIdx.x == gridDim.x - 1;
    const uint32_t ntile = (uint32_t)((r_end - r_begin + kRows - 1) / kRows);
    const uint32_t nitems = ntile * kMats * p.nitem;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1;

    if (tid == 0) {
        prefetch_tmap(last_cta ? &p.wmap_last : &p.wmap_main);
        prefetch_tmap(last_cta ? &p.smap_last : &p.smap_main);
        if (kMats == 2) {
            prefetch_tmap(last_cta ? &p.wmap2_last : &p.wmap2_main);
            prefetch_tmap(last_cta ? &p.smap2_last : &p.smap2_main);
        }
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        *failed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    const uint32_t pre = p.pre_issue < ring_to ? p.pre_issue : ring_to;
    if (tid == 0) {
        // weights are read-only parameters: a few items before the dependency wait
        for (uint32_t i = 0; i < pre; ++i) issue_item<kMats>(p, smem, i, last_cta);
    }
    // rotation tasks (matrix, block): one rotation per block, or two when the
    // fused matrices have different signs; warp pair pr takes tasks pr, pr + nrot, ...
    const uint32_t nrmat = (kMats == 2 && p.signs2 != p.signs) ? 2 : 1;
    const uint32_t ntask = nrmat * p.nblk;
    const uint32_t nrot = ntask < kRotPairs ? ntask : kRotPairs;
    const uint32_t pr = warp >> 1;
    const int t = tid & 63;
    auto task_src = [&](uint32_t task) {
        return XSource{p.x, task >= p.nblk ? p.signs2 : p.signs, p.k, p.x_dtype};
    };
    float d[16];
    if (pr < nrot) {
        const XSource xs0 = task_src(pr);
        if (xs0.signs) load_signs16(xs0, pr % p.nblk, t, d);     // also read-only
    }
    pdl_launch_dependents();
    pdl_wait();          // x may come from the preceding kernel

    float v[16];
    if (pr < nrot) load_run16(task_src(pr), pr % p.nblk, t, v);
    __syncthreads();     // every warp's x request is out: the rest of the ring queues behind them
    if (tid == 0) {
        for (uint32_t i = pre; i < ring_to; ++i) issue_item<kMats>(p, smem, i, last_cta);
        *issued = ring_to;
    }
    uint8_t *act_s = smem + p.off_act;
    if (pr < nrot) {
        float *tile = reinterpret_cast<float *>(smem + p.off_part + pr * kRotScratch);
        for (uint32_t task = pr; task < ntask; task += nrot) {
            const XSource xs = task_src(task);
            const uint32_t b = task % p.nblk;
            if (task != pr) {
                if (xs.signs) load_signs16(xs, b, t, d);
                load_run16(xs, b, t, v);
            }
            int E;
            const int16_t *qs = rotate_quantize16(xs.signs != nullptr, t, v, d, tile, 1 + pr, &E);
            pack_pq2(qs, act_s + (task / p.nblk) * p.act_bytes, p.groups, b, t, E, 1 + pr);
        }
    }
    __syncthreads();

    bool ok = true;
    // group gw of the item = 16-byte chunks 2gi, 2gi+1 of column h's 128-byte
    // line; this warp reads chunk 2gi + half (words 4 half .. 4 half + 3), swizzled by row % 8
    const uint32_t gw = warp & 7, half = warp >> 3, h = gw >> 2, gi = gw & 3;
    const uint32_t ch = ((2 * gi + half) ^ (lane & 7)) << 4;
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    const bool refill = nitems > p.nslots;    // otherwise the whole slice sits in the ring
    uint32_t slot = 0, phase = 0, item = 0;
    for (uint32_t tile = 0; tile < ntile; ++tile) {
        float y[kMats][4];      // rows lane + 32q of the tile, per matrix
#pragma unroll
        for (int mt = 0; mt < kMats; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q) y[mt][q] = 0.f;
        for (uint32_t jj = 0; jj < kMats * p.nitem; ++jj, ++item) {
            const uint32_t mat = kMats == 1 ? 0 : (jj >= p.nitem), j = jj - mat * p.nitem;
            const uint8_t *act_m = act_s + (mat < nrmat ? mat : 0) * p.act_bytes;
            const float2 *gs = reinterpret_cast<const float2 *>(act_m + p.groups * 256);
            ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err);
            const uint32_t G = j * 8 + gw;
            if (ok && G < p.groups) {
                const uint8_t *sa = smem + p.off_ring + slot * kItemBytes;
                const uint8_t *wr = sa + h * kBoxBytes + lane * 128 + ch;
                uint32_t w[4][4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(wr + q * 4096);
                    w[q][0] = a.x; w[q][1] = a.y; w[q][2] = a.z; w[q][3] = a.w;
                }
                const uint4 *aw = reinterpret_cast<const uint4 *>(act_m + (uint64_t)G * 256 + half * 128);
                int acc[4][4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int t = 0; t < 4; ++t) acc[q][t] = 0;
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint4 lo = aw[2 * wi], hi = aw[2 * wi + 1];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t c = w[q][wi];
                        acc[q][0] = dp2a_hi(hi.x, c & 0x03030303u, dp2a_lo(lo.x, c & 0x03030303u, acc[q][0]));
                        acc[q][1] = dp2a_hi(hi.y, c & 0x0C0C0C0Cu, dp2a_lo(lo.y, c & 0x0C0C0C0Cu, acc[q][1]));
                        acc[q][2] = dp2a_hi(hi.z, c & 0x30303030u, dp2a_lo(lo.z, c & 0x30303030u, acc[q][2]));
                        acc[q][3] = dp2a_hi(hi.w, c & 0xC0C0C0C0u, dp2a_lo(lo.w, c & 0xC0C0C0C0u, acc[q][3]));
                    }
                }
                const float2 f = gs[G];
                const int off = half ? 0 : __float_as_int(f.y);     // the group's sum of x16, once
                // scale box: row r at r * 16 bytes holds the item's 8 scales
                const uint8_t *sc = sa + 2 * kBoxBytes + lane * 16 + 2 * gw;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = acc[q][0] + (acc[q][1] >> 2) + (acc[q][2] >> 4) + (acc[q][3] >> 6) - off;
                    const float s = __half2float(*reinterpret_cast<const __half *>(sc + q * 512));
                    if (kMats == 1 || mat == 0) y[0][q] = fmaf(s * f.x, (float)t, y[0][q]);
                    else y[kMats - 1][q] = fmaf(s * f.x, (float)t, y[kMats - 1][q]);
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
                        if (ok && !*(volatile uint32_t *)failed && item + p.nslots < nitems) {
                            fence_proxy_async();
                            issue_item<kMats>(p, smem, item + p.nslots, last_cta);
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
        }
#pragma unroll
        for (int mt = 0; mt < kMats; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q) part[(mt * kWarps + warp) * kRows + 32 * q + lane] = y[mt][q];
        __syncthreads();
        if (warp < kRows / 32) {
            const uint32_t rl = warp * 32 + lane;
            const uint64_t r = r_begin + (uint64_t)tile * kRows + rl;
            float acc[kMats];
#pragma unroll
            for (int mt = 0; mt < kMats; ++mt) {
                acc[mt] = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) acc[mt] += part[(mt * kWarps + w) * kRows + rl];
            }
            // fused gate/up: SwiGLU, silu(g) * u with silu(g) = g / (1 + e^-g)
            const float out = kMats == 1 ? acc[0] : acc[0] / (1.f + expf(-acc[0])) * acc[kMats - 1];
            if (r < r_end) store1(p.y, r, p.y_dtype, out);
        }
        __syncthreads();
    }
    // after a timed-out wait: let the copies still in flight land (at most one
    // per slot, the last one issued into it) before the CTA's memory is freed
    if (tid == 0 && *(volatile uint32_t *)failed) {
        const uint32_t n_issued = *(volatile uint32_t *)issued;
        for (uint32_t i = n_issued > p.nslots ? n_issued - p.nslots : 0; i < n_issued; ++i)
            mbar_wait(bar0 + 8 * (i % p.nslots), (i / p.nslots) & 1, p.err, 200000000ll);
    }
}

}  // namespace

bool gemv_pq2_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                       IntPlan *plan, int mats, bool two_rotations) {
    *plan = IntPlan{};
    if (M != 1 || mats < 1 || mats > 2) return false;
    if (rotate && g.k % 1024) return false;
    // scale rows must be whole 16-byte units (8 groups) for the scale boxes
    if (g.scale_row_bytes % 16 || g.base_row_bytes % 16 || g.payload_bytes % 16) return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31)) return false;
    const uint32_t groups = (uint32_t)g.groups_per_row;
    const uint32_t act_one = ((groups * 264 + 15) / 16) * 16;
    const uint32_t nrmat = (mats == 2 && two_rotations) ? 2 : 1;
    const uint32_t act_bytes = nrmat * act_one;
    // tile partial sums, and before them the rotation's scratch (one padded tile per rotating warp pair)
    const uint32_t nrot = std::min<uint32_t>(nrmat * (uint32_t)((g.k + 1023) / 1024), kRotPairs);
    const uint32_t part_bytes = std::max<uint32_t>(mats * kWarps * kRows * 4, nrot * kRotScratch);
    const uint32_t bar_bytes = kMaxSlots * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 4) * 4;
    const uint32_t fixed = act_bytes + part_bytes + bar_bytes + cnt_bytes;
    if ((int)fixed + 2 * (int)kItemBytes > smem_limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((smem_limit - (int)fixed) / (int)kItemBytes));
    // one CTA per SM with ~n / SMs rows each
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)sms, g.n / 64));
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid = (g.n + R - 1) / R;
    plan->ok = true;
    plan->mats = mats;
    plan->act_one = act_one;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nitem = (groups + 7) / 8;
    plan->nslots = nslots;
    plan->pre_issue = std::min<uint32_t>(1, nslots);
    plan->off_ring = 0;
    plan->off_act = nslots * kItemBytes;
    plan->off_part = plan->off_act + act_bytes;
    plan->off_bar = plan->off_part + part_bytes;
    plan->off_cnt = plan->off_bar + bar_bytes;
    plan->smem = plan->off_cnt + cnt_bytes;
    plan->workspace = 0;
    return true;
}

int gemv_pq2_int_launch(const IntPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                        int x_dtype, const uint16_t *signs, void *y, int y_dtype, cudaStream_t stream, bool pdl,
                        const uint8_t *payload2, const uint16_t *signs2) {
    IntParams p;
    std::memset(&p, 0, sizeof p);
    const uint8_t *base = payload + g.base_offset, *scale = payload + g.scale_offset;
    p.x = x;
    p.signs = signs;
    p.signs2 = plan.mats == 2 ? signs2 : signs;
    p.act_bytes = plan.act_one;
    p.y = y;
    p.n = g.n;
    p.k = (uint32_t)g.k;
    p.groups = (uint32_t)g.groups_per_row;
    p.nblk = (uint32_t)((g.k + 1023) / 1024);
    p.nitem = plan.nitem;
    p.rows_per_cta = plan.rows_per_cta;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.pre_issue = plan.pre_issue;
    p.off_ring = plan.off_ring;
    p.off_act = plan.off_act;
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
    if (plan.mats == 2) {
        // the second matrix: same geometry, its own payload
        const uint8_t *base2 = payload2 + g.base_offset, *scale2 = payload2 + g.scale_offset;
        if (G > 1) {
            st = encode_row_tiles(&p.wmap2_main, base2, g.base_row_bytes, R, G - 1, 128, kRows, true);
            if (!st) st = encode_row_tiles(&p.smap2_main, scale2, g.scale_row_bytes, R, G - 1, 16, kRows, false);
            if (st) return st;
        }
        st = encode_rows(&p.wmap2_last, base2 + (G - 1) * R * g.base_row_bytes, g.base_row_bytes, last_rows, 128,
                         kRows, true);
        if (!st)
            st = encode_rows(&p.smap2_last, scale2 + (G - 1) * R * g.scale_row_bytes, g.scale_row_bytes, last_rows,
                             16, kRows, false);
        if (st) return st;
    }
    auto kernel = plan.mats == 2 ? gemv_pq2_int_kernel<2> : gemv_pq2_int_kernel<1>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
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
    e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
