// Decode GEMV for PTQ1_0_G128 weights and one activation row (M = 1), on the
// CUDA cores' integer pipes, with the activation rotation fused in.
//
// What it computes:
//   y[r] = sum_g scale[r][g] * sum_{j<128} (t[r][128g+j] - 1) * xr[128g+j]
// with xr the forward-rotated activation (per 1024-block H (D * x) / 32,
// "artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2) and t
// the base-3 digits of the planes ("bonsai三元GGUF模型转ninfer模型01" §3-§4): base
// byte j of a group holds weights 5j .. 5j+4 as (byte / 3^i) % 3, high byte h
// holds weights 120 + 4h .. 123 + 4h; one binary16 scale per group.
//
// Work split: a CTA owns a contiguous range of rows. When its eight warp pairs
// could not rotate all 1024-blocks of k in one round, two or four CTAs of a
// cluster share a row range and split its groups: each rotates and reads only
// its share, and the partial row sums meet through distributed shared memory at
// the end (rank r finishes the r-th part of the rows, adding the ranks' sums in
// rank order).
//
// Activation: a warp pair rotates each of the CTA's blocks and rounds it to
// 16-bit fixed point (rot2.cuh: x16 = rint(xr * 2^E'), max |x16| < 2^14), then
// packs, per group, 64 operand words: for base byte
// j (< 24), (x16[5j], x16[5j+1]) and (x16[5j+2], x16[5j+3]); for the four bytes
// 4q .. 4q+3, the pairs of their fifth weights (x16[5(4q+2c)+4],
// x16[5(4q+2c+1)+4]); for high byte h, its two pairs; and one group entry
// {2^-E (with the transform's 1/32), sum of the group's x16}.
//
// Thread mapping: thread t owns group t % nG of the CTA's nG
// groups for the whole launch, holding its 64 operand words in registers, and
// row set t / nG. Weights arrive in batches of nsets * u rows as tensor boxes
// of 8-byte elements, each plane seen as {row, rows, row ranges}: the CTA's
// base bytes of the batch's rows in one box per wg groups (wg <= 84, so that a
// box row stays within 256 elements), then their high bytes and their scales
// (one box each, rounded out to whole 16-byte units). The boxes land row-major
// in a slot of a shared-memory ring, so that the lanes of a warp read
// consecutive groups of one row, without bank conflicts. Per row a
// thread writes one partial sum to the slot's partial buffer (group-major, an
// odd number of floats per group). Once every math warp has finished a batch,
// its partials are added per row, y (or the CTA's share of it) stored and the
// slot refilled: by warp 15 when it has no group of its own (it shares a
// scheduler with fewer math warps), else by the warps in turn, each after its
// own next batch. Only the first batch is requested before the
// programmatic-dependent-launch wait: that wait returns only once memory
// requests already in flight have landed.
//
// Arithmetic: a 256-entry table maps a code byte to its digits as bytes
// (t0 | t1 << 8 | t2 << 16 | t3 << 24) with t4 in bits 2-3 of byte 0, and in
// its second half the same with t4 in bits 2-3 of byte 1; entry B at B * 256,
// each half held once per lane (lane l's copy at + 4 l, bank l), so that a
// byte permute of the code word and 4 l (or 4 l + 128) forms a lane's address
// in one instruction. Per base byte dp2a multiplies (t0, t1) and (t2, t3) by
// their activation pairs; bytes 0 and 2 of a code word look up the first half,
// bytes 1 and 3 the second, so that two or-and operations and one byte permute
// gather the t4 fields of the word's four bytes, multiplied by their pairs
// (times 4, removed at the end); all exact in int32. Per group:
//   y += scale * 2^-E * (sum t x16 - sum x16)                    (value = t - 1)
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "act16.cuh"
#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"
#include "rot2.cuh"

namespace ninfer {
namespace {

constexpr int kThreads = 512;              // four warps per scheduler: up to 128 registers a thread
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kMaxSlots = 12;
constexpr uint32_t kActWords = 64;
// Groups sit kActStride words apart: 17 16-byte units, an odd number, so that
// lanes loading consecutive groups' words meet no bank conflicts.
constexpr uint32_t kActStride = 68;
static_assert(kActStride >= kActWords && kActStride % 8 == 4, "operand words: an odd number of 16-byte units");
constexpr uint32_t kActGroupBytes = kActStride * 4;
constexpr uint32_t kLutStride = 256;        // entry B at B * 256: 32 lane copies of each half
constexpr uint32_t kLutBytes = 256 * kLutStride;
constexpr uint32_t kPairs = kWarps / 2;     // rotating warp pairs; named barriers 1 .. 8
constexpr uint32_t kBarPair0 = 1;
// the table, and before it the pairs' rotation scratch, start the shared memory
constexpr uint32_t kRegion0 = (kPairs * kRotScratchBytes > kLutBytes ? kPairs * kRotScratchBytes : kLutBytes);
static_assert(kRegion0 % 128 == 0, "ring slots 128-byte aligned");
static_assert(kBarPair0 + kPairs <= 16, "named barriers");
constexpr uint32_t kMaxClusterRows = 4096;  // rows of a split range (their partial sums stay in shared memory)
// after the full and empty barriers of the slots: the failure flag, then per slot
// the last batch issued into it
constexpr uint32_t kFlagWords = 1 + kMaxSlots;
constexpr uint32_t kBarBytes = (2 * kMaxSlots * 8 + 4 * kFlagWords + 15) / 16 * 16;

struct Ptq1Params {
    // planes as 8-byte elements {row, rows, row ranges}: every row range but the
    // last, and the last
    CUtensorMap bmap_main, bmap_last, hmap_main, hmap_last, smap_main, smap_last;
    const void *x;
    const uint16_t *signs;
    void *y;
    uint64_t n;
    uint32_t units;                 // row ranges (CTAs, or CTA pairs when clustered)
    uint32_t k, groups;
    uint32_t rows_per_cta;          // rows of a CTA (of a cluster when clustered)
    uint32_t hbytes;                // high bytes (and scales) per row in a slot: the same for every rank
    uint32_t nsets, u;              // row sets and rows per set of a batch
    uint32_t wg, nbx, bstride;      // groups per base box, base boxes per batch, their distance in a slot
    uint32_t nslots, nslots_inv, pre_issue;
    uint32_t slot_bytes, slot_high, slot_scale;         // slot size and the offsets of its high / scale regions
    uint32_t part_stride, part_slot_bytes;
    uint32_t off_ring, off_part, off_rs, off_bar;       // table / rotation scratch at 0; operand words at off_part
    int x_dtype, y_dtype;
    uint32_t *err;
    long long wait_cycles;
};

// This CTA's share: row range unit (rows [r0, r0 + rows)), groups [g0, g0 + ng),
// high bytes and scales of groups [h0, h0 + hbytes / 2) (a slot holds the plan's
// width from h0, which covers them).
struct Cta {
    uint64_t r0;
    uint32_t unit, rows, g0, ng, h0, hbytes, nbatch;
};

__device__ __forceinline__ Cta cta_share(const Ptq1Params &p, uint32_t csize, uint32_t crank) {
    Cta c;
    c.unit = blockIdx.x / csize;
    c.r0 = (uint64_t)c.unit * p.rows_per_cta;
    const uint64_t left = c.r0 < p.n ? p.n - c.r0 : 0;
    c.rows = left < p.rows_per_cta ? (uint32_t)left : p.rows_per_cta;
    // rank r of C: groups [s_r, s_{r+1}), s_r = floor(r G / C) rounded down to even
    auto split = [&](uint32_t r) { return r >= csize ? p.groups : ((r * p.groups) / csize) & ~1u; };
    c.g0 = split(crank);
    c.ng = split(crank + 1) - c.g0;
    c.h0 = c.g0 & ~7u;
    c.hbytes = 2 * (((c.g0 + c.ng + 7) & ~7u) - c.h0);
    const uint32_t br = p.nsets * p.u;
    c.nbatch = (c.rows + br - 1) / br;
    return c;
}

__device__ __forceinline__ uint32_t slot_of(uint32_t b, uint32_t nslots, uint32_t inv, uint32_t &phase) {
    const uint32_t cycle = __umulhi(b, inv);     // b / nslots (b < 2^29)
    phase = cycle & 1;
    return b - cycle * nslots;
}

// Batch b's rows into its ring slot (one thread). Rows past the range read as
// zero and cost no traffic; the transaction counts whole boxes.
__device__ __forceinline__ void issue_batch(const Ptq1Params &p, const Cta &c, uint8_t *smem, uint32_t b) {
    const uint32_t br = p.nsets * p.u;
    uint32_t phase;
    const uint32_t slot = slot_of(b, p.nslots, p.nslots_inv, phase);
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, br * (24 * p.wg * p.nbx + 2 * p.hbytes));
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * p.slot_bytes;
    const bool last = c.unit == p.units - 1;
    const int y = (int)(b * br), z = last ? 0 : (int)c.unit;
    for (uint32_t bx = 0; bx < p.nbx; ++bx)
        tma_load_3d(dst + bx * p.bstride, last ? &p.bmap_last : &p.bmap_main, (int)(3 * (c.g0 + bx * p.wg)), y, z, bar);
    tma_load_3d(dst + p.slot_high, last ? &p.hmap_last : &p.hmap_main, (int)(c.h0 / 4), y, z, bar);
    tma_load_3d(dst + p.slot_scale, last ? &p.smap_last : &p.smap_main, (int)(c.h0 / 4), y, z, bar);
}

// Rotates block b with the pair and writes the operand words and group entries
// {2^-E (with the transform's 1/32), sum of the group's x16 (int bits)} of those
// of its eight groups that lie in [g0, g0 + ng) (local index G - g0).
__device__ __forceinline__ void rotate_pack(bool rotate, float (&v)[16], const float (&d)[16], uint32_t b,
                                            uint32_t g0, uint32_t ng, uint8_t *act, float *scr, int t, uint32_t bar) {
    const int lane = t & 31;
    uint32_t qb[16];
    const int E = rotate_quant2(rotate, v, d, scr, t, bar, qb);
    const float f = ldexpf(1.f, -E - (rotate ? 5 : 0));
    // x16 in natural order (int16) in the scratch: elements 512 i + 8 t .. + 7
    int16_t *qs = reinterpret_cast<int16_t *>(scr);
    float2 *gs = reinterpret_cast<float2 *>(act + ng * kActGroupBytes);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t *q = qb + 8 * i;
        uint4 w;
        w.x = __byte_perm(q[0], q[1], 0x5410);
        w.y = __byte_perm(q[2], q[3], 0x5410);
        w.z = __byte_perm(q[4], q[5], 0x5410);
        w.w = __byte_perm(q[6], q[7], 0x5410);
        *reinterpret_cast<uint4 *>(qs + 512 * i + 8 * t) = w;
        // the group's sum of x16 (group 4 i + t / 16 of the block): the 16 lanes of each half-warp
        const int sum = (int)(q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7] - 8u * 0x4B400000u);
        const int s_lo = __reduce_add_sync(0xffffffffu, lane < 16 ? sum : 0);
        const int s_hi = __reduce_add_sync(0xffffffffu, lane < 16 ? 0 : sum);
        const uint32_t L = b * 8 + 4 * i + (t >> 4) - g0;     // wraps past ng when below g0
        if ((lane & 15) == 0 && L < ng) gs[L] = make_float2(f, __int_as_float(lane < 16 ? s_lo : s_hi));
    }
    named_barrier(bar, 64);
    // operand words: the block's 8 groups have 208 code bytes (192 base, 16 high);
    // thread t takes bytes t, t + 64, t + 128 and t + 192
    uint32_t *aw = reinterpret_cast<uint32_t *>(act);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = t + 64 * i;
        if (u >= 208) break;
        const uint32_t gl = u < 192 ? u / 24 : (u - 192) >> 1, L = b * 8 + gl - g0;
        if (L >= ng) continue;
        uint32_t *dst = aw + L * kActStride;
        if (u < 192) {
            const uint32_t j = u % 24;
            const int16_t *e = qs + 128 * gl + 5 * j;
            dst[2 * j] = (uint32_t)(uint16_t)e[0] | ((uint32_t)(uint16_t)e[1] << 16);
            dst[2 * j + 1] = (uint32_t)(uint16_t)e[2] | ((uint32_t)(uint16_t)e[3] << 16);
            reinterpret_cast<int16_t *>(dst + 48 + 2 * (j >> 2) + ((j >> 1) & 1))[j & 1] = e[4];
        } else {
            const uint32_t hh = (u - 192) & 1;
            const int16_t *e = qs + 128 * gl + 120 + 4 * hh;
            dst[60 + 2 * hh] = (uint32_t)(uint16_t)e[0] | ((uint32_t)(uint16_t)e[1] << 16);
            dst[61 + 2 * hh] = (uint32_t)(uint16_t)e[2] | ((uint32_t)(uint16_t)e[3] << 16);
        }
    }
    named_barrier(bar, 64);      // the scratch may be reused
}

// Lane's copy of the table entry of byte c of w: lut + (B_c << 8 | lane4), lane4
// = 4 lane (first half) or 4 lane + 128 (second half).
__device__ __forceinline__ uint32_t lut_entry(const uint8_t *lut, uint32_t w, uint32_t lane4, uint32_t c) {
    return *reinterpret_cast<const uint32_t *>(lut + __byte_perm(w, lane4, 0x5504u | (c << 4)));
}

// sum_j t_j x16_j over the group's six base words (four code bytes each) and
// two high bytes, from the operand words av (the pairs of base byte j at 2 j,
// the fifth-weight pairs of word q at 48 + 2 q, the pairs of high byte h at
// 60 + 2 h).
__device__ __forceinline__ int group_dot(const uint32_t (&bw)[6], uint32_t hb, const uint8_t *lut, uint32_t lane4,
                                         const uint32_t (&av)[kActWords]) {
    int acc[4] = {0, 0, 0, 0}, acc4 = 0;
    const uint32_t lane4b = lane4 | 128u;
#pragma unroll
    for (int q = 0; q < 6; ++q) {
        uint32_t W[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) W[c] = lut_entry(lut, bw[q], (c & 1) ? lane4b : lane4, c);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t m = W[c] & 0x03030303u;
            const int j = 4 * q + c;
            acc[c] = dp2a_lo(av[2 * j], m, acc[c]);
            acc[c] = dp2a_hi(av[2 * j + 1], m, acc[c]);
        }
        // 4 * t4 sits in bits 2-3 of byte 0 (bytes 0, 2) or byte 1 (bytes 1, 3):
        // gather the four into bytes 0-3
        const uint32_t g = __byte_perm((W[0] | W[1]) & 0x0C0Cu, (W[2] | W[3]) & 0x0C0Cu, 0x5410u);
        acc4 = dp2a_lo(av[48 + 2 * q], g, acc4);
        acc4 = dp2a_hi(av[49 + 2 * q], g, acc4);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t m = lut_entry(lut, hb, lane4, h) & 0x03030303u;
        acc[h] = dp2a_lo(av[60 + 2 * h], m, acc[h]);
        acc[h] = dp2a_hi(av[61 + 2 * h], m, acc[h]);
    }
    return acc[0] + acc[1] + acc[2] + acc[3] + (acc4 >> 2);
}

// kU: rows per row set of a batch (p.u), 1 or 2, fixed per instance so that the
// row loop unrolls
template <int kXType, int kU>
__global__ void __launch_bounds__(kThreads, 1) gemv_ptq1_int_kernel(const __grid_constant__ Ptq1Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t csize = cluster_nctarank(), crank = csize > 1 ? cluster_ctarank() : 0u;
    const Cta c = cta_share(p, csize, crank);
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t empty0 = bar0 + 8 * kMaxSlots;
    uint32_t *failed = reinterpret_cast<uint32_t *>(smem + p.off_bar + 16 * kMaxSlots);
    uint32_t *lastb = failed + 1;               // per slot: the last batch issued into it
    uint8_t *act = smem + p.off_part;           // operand words, later the partial sums
    const uint32_t nact = p.nsets * c.ng;        // threads with a group
    const uint32_t nmw = (nact + 31) / 32;       // warps with work
    const uint32_t ring_to = min(p.nslots, c.nbatch);
    const uint32_t pre = min(p.pre_issue, ring_to);

    if (csize == 2) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (tid == 0) {
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, nmw);
            lastb[s] = s;
        }
        *failed = 0;
        fence_mbar_init();
        const bool last = c.unit == p.units - 1;
        prefetch_tmap(last ? &p.bmap_last : &p.bmap_main);
        prefetch_tmap(last ? &p.hmap_last : &p.hmap_main);
        prefetch_tmap(last ? &p.smap_last : &p.smap_main);
        // weights are read-only parameters: the first batches before the dependency wait
        for (uint32_t b = 0; b < pre; ++b) issue_batch(p, c, smem, b);
    }

    // rotation: pair pr takes blocks first + pr, first + pr + 8, ...
    const uint32_t b_first = c.g0 / 8;
    const uint32_t nblk = c.ng ? (c.g0 + c.ng - 1) / 8 - b_first + 1 : 0u;
    const uint32_t pr = (uint32_t)warp >> 1;
    const int t = tid & 63;
    float v[16], d[16];
    if (pr < nblk && p.signs) load_signs2(p.signs, b_first + pr, t, d);      // read-only
    pdl_launch_dependents();
    pdl_wait();          // x may come from the preceding kernel; y may still be read by it
    if (tid == 0)
        for (uint32_t b = pre; b < ring_to; ++b) issue_batch(p, c, smem, b);
#pragma unroll 1
    for (uint32_t task = pr; task < nblk; task += kPairs) {
        const uint32_t b = b_first + task;
        if (task != pr && p.signs) load_signs2(p.signs, b, t, d);
        load_block2<kXType>(p.x, p.k, b, t, v);
        rotate_pack(p.signs != nullptr, v, d, b, c.g0, c.ng, act, reinterpret_cast<float *>(smem + pr * kRotScratchBytes),
                    t, kBarPair0 + pr);
    }
    __syncthreads();     // operand words complete; the rotation scratch is free for the table
    {
        // digit table: thread t builds half t % 2 of entry t / 2 (512 threads, 512
        // halves) as eight 16-byte stores of 4 lane copies each, in an order
        // staggered by lane so that a warp's stores spread over all banks
        static_assert(kThreads == 512, "one table half per thread");
        uint32_t B = (uint32_t)tid >> 1, W = 0;
        const uint32_t half = (uint32_t)tid & 1;
#pragma unroll
        for (int e = 0; e < 5; ++e) {
            const uint32_t dg = B % 3;
            B /= 3;
            W |= e < 4 ? dg << (8 * e) : dg << (2 + 8 * half);
        }
        uint8_t *ent = smem + ((uint32_t)tid >> 1) * kLutStride + 128 * half;
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) *reinterpret_cast<uint4 *>(ent + 16 * ((k2 + lane) & 7)) = make_uint4(W, W, W, W);
    }
    const bool math = (uint32_t)tid < nact;
    const uint32_t gl = math ? (uint32_t)tid % c.ng : 0u, set = math ? (uint32_t)tid / c.ng : 0u;
    uint32_t av[kActWords];
    float fx = 0.f;
    int off = 0;
    if (math) {
        const uint4 *src = reinterpret_cast<const uint4 *>(act + gl * kActGroupBytes);
#pragma unroll
        for (int i = 0; i < (int)kActWords / 4; ++i) {
            const uint4 a = src[i];
            av[4 * i] = a.x;
            av[4 * i + 1] = a.y;
            av[4 * i + 2] = a.z;
            av[4 * i + 3] = a.w;
        }
        const float2 e = reinterpret_cast<const float2 *>(act + c.ng * kActGroupBytes)[gl];
        fx = e.x;
        off = __float_as_int(e.y);
    }
    __syncthreads();     // table built; the operand-word area now takes the partial sums

    bool ok = true;
    const uint32_t br = p.nsets * p.u;
    float *rs = reinterpret_cast<float *>(smem + p.off_rs);     // this CTA's row sums (split ranges)
    // batch b, once every warp is done with it: its row sums over the CTA's groups
    // (lanes = rows), then the slot's refill with batch b + nslots
    auto reduce = [&](uint32_t b) {
        uint32_t phase;
        const uint32_t slot = slot_of(b, p.nslots, p.nslots_inv, phase);
        const uint32_t rows_b = min(br, c.rows - b * br);
        ok = ok && mbar_wait(empty0 + 8 * slot, phase, p.err, p.wait_cycles);
        if (ok) {
            const float *part = reinterpret_cast<const float *>(smem + p.off_part + slot * p.part_slot_bytes);
            for (uint32_t rr = lane; rr < rows_b; rr += 32) {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                uint32_t g = 0;
                for (; g + 4 <= c.ng; g += 4) {
                    a0 += part[g * p.part_stride + rr];
                    a1 += part[(g + 1) * p.part_stride + rr];
                    a2 += part[(g + 2) * p.part_stride + rr];
                    a3 += part[(g + 3) * p.part_stride + rr];
                }
                for (; g < c.ng; ++g) a0 += part[g * p.part_stride + rr];
                const float acc = (a0 + a1) + (a2 + a3);
                const uint32_t row = b * br + rr;
                if (csize > 1) rs[row] = acc;
                else store1(p.y, c.r0 + row, p.y_dtype, acc);
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (!ok) {
                *failed = 1;
            } else if (!*(volatile uint32_t *)failed && b + p.nslots < c.nbatch) {
                fence_proxy_async();
                lastb[slot] = b + p.nslots;
                issue_batch(p, c, smem, b + p.nslots);
            }
        }
        __syncwarp();
    };
    const bool dedicated = nmw < (uint32_t)kWarps;     // warp kWarps - 1 adds the partials
    if ((uint32_t)warp < nmw) {
        const uint32_t lane4 = 4u * (uint32_t)lane;
        // group gl: box gl / wg, bytes 24 (gl % wg) of each of its rows
        const uint32_t rb_b = 24 * p.wg, o_b = (gl / p.wg) * p.bstride + 24 * (gl % p.wg);
        const uint32_t o_h = p.slot_high + 2 * (c.g0 + gl - c.h0), o_s = p.slot_scale + 2 * (c.g0 + gl - c.h0);
#pragma unroll 1
        for (uint32_t b = 0; b < c.nbatch; ++b) {
            uint32_t phase;
            const uint32_t slot = slot_of(b, p.nslots, p.nslots_inv, phase);
            const uint32_t rows_b = min(br, c.rows - b * br);
            ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err, p.wait_cycles);
            if (ok && math) {
                const uint8_t *sa = smem + p.off_ring + slot * p.slot_bytes;
                float *part = reinterpret_cast<float *>(smem + p.off_part + slot * p.part_slot_bytes) + gl * p.part_stride;
#pragma unroll
                for (uint32_t i = 0; i < (uint32_t)kU; ++i) {
                    const uint32_t rb = i * p.nsets + set;
                    if (rb >= rows_b) break;
                    const uint8_t *row = sa + rb * rb_b + o_b;
                    const uint2 b0 = *reinterpret_cast<const uint2 *>(row);
                    const uint2 b1 = *reinterpret_cast<const uint2 *>(row + 8);
                    const uint2 b2 = *reinterpret_cast<const uint2 *>(row + 16);
                    const uint32_t bw[6] = {b0.x, b0.y, b1.x, b1.y, b2.x, b2.y};
                    const uint32_t hb = *reinterpret_cast<const uint16_t *>(sa + rb * p.hbytes + o_h);
                    const float s = __half2float(*reinterpret_cast<const __half *>(sa + rb * p.hbytes + o_s));
                    const int dot = group_dot(bw, hb, smem, lane4, av);
                    part[rb] = (s * fx) * (float)(dot - off);
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (!ok) *failed = 1;
                mbar_arrive(empty0 + 8 * slot);
            }
            // warps take the batches' sums in turn, one batch behind their own work
            if (!dedicated && b >= 1 && (b - 1) % nmw == (uint32_t)warp) reduce(b - 1);
        }
        if (!dedicated && c.nbatch >= 1 && (c.nbatch - 1) % nmw == (uint32_t)warp) reduce(c.nbatch - 1);
    } else if (dedicated && warp == kWarps - 1) {
#pragma unroll 1
        for (uint32_t b = 0; b < c.nbatch; ++b) reduce(b);
    }
    __syncthreads();     // every row sum is in place; failures are recorded

    if (csize > 1) {
        // rows split in csize parts of rq rows (a multiple of 4); rank q finishes
        // part q: warp q stores this rank's sums for part q, four rows per store,
        // in rank q's inbox (rows_per_cta rounded up to 4 floats after the row
        // sums: csize arrays of rq floats, one per source rank)
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");     // every CTA of the cluster is running
        const uint32_t rq = ((c.rows + csize - 1) / csize + 3) & ~3u;
        float *inbox = rs + ((p.rows_per_cta + 3) & ~3u);
        if ((uint32_t)warp < csize) {
            const uint32_t q = warp;
            const uint32_t peer = mapa_shared(smem_u32(inbox + crank * rq), q);
            const uint32_t lo = q * rq, hi = min(c.rows, lo + rq);
            for (uint32_t r4 = lo + 4 * lane; r4 < hi; r4 += 128) {
                // rows past hi (at most 3, within the rounding) are sent but never read
                const float4 v = *reinterpret_cast<const float4 *>(rs + r4);
                st_cluster_v4(peer + 4 * (r4 - lo), make_uint4(__float_as_uint(v.x), __float_as_uint(v.y),
                                                              __float_as_uint(v.z), __float_as_uint(v.w)));
            }
        }
        cluster_sync();
        const uint32_t lo = crank * rq, hi = min(c.rows, lo + rq);
        for (uint32_t rr = lo + tid; rr < hi; rr += kThreads) {
            float acc = 0.f;
            for (uint32_t s2 = 0; s2 < csize; ++s2) acc += inbox[s2 * rq + (rr - lo)];      // rank order
            store1(p.y, c.r0 + rr, p.y_dtype, acc);
        }
    }
    // after a timed-out wait: let the copies still in flight land (the last one
    // issued into each slot) before the CTA's memory is freed
    if (tid == 0 && *(volatile uint32_t *)failed) {
        for (uint32_t s = 0; s < ring_to; ++s)
            mbar_wait(bar0 + 8 * s, (lastb[s] / p.nslots) & 1, p.err, 200000000ll);
    }
}

// Clusters of C CTAs (one per SM) that can be resident at once, from the
// occupancy calculator, once per device and C; sms / C if it cannot tell.
uint32_t max_clusters(uint32_t C, int smem_limit, int sms) {
    static std::mutex mu;
    static int cache[64][5];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return (uint32_t)sms / C;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev][C] > 0) return (uint32_t)cache[dev][C];
    int n = 0;
    const void *kernel = (const void *)gemv_ptq1_int_kernel<NINFER_BF16, 2>;
    if (set_smem_attribute(kernel, smem_limit) == NINFER_OK) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * ((uint32_t)sms / C));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = (size_t)smem_limit;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, (void (*)(Ptq1Params))gemv_ptq1_int_kernel<NINFER_BF16, 2>, &cfg) !=
            cudaSuccess)
            n = 0;
        (void)cudaGetLastError();
    }
    if (n <= 0) n = sms / (int)C;
    n = std::min(n, sms / (int)C);
    cache[dev][C] = n;
    return (uint32_t)n;
}

}  // namespace

bool gemv_ptq1_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                        Ptq1Plan *plan) {
    *plan = Ptq1Plan{};
    if (M != 1 || sms < 2) return false;
    if (rotate && g.k % 1024) return false;
    // high and scale rows are whole 16-byte units (8 groups), as every copied segment is
    if (g.groups_per_row % 8 || g.base_row_bytes % 16 || g.high_row_bytes % 16 || g.scale_row_bytes % 16) return false;
    if (g.base_offset % 16 || g.high_offset % 16 || g.scale_offset % 16) return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31) || g.n == 0) return false;
    const uint32_t G = (uint32_t)g.groups_per_row;
    // the ranks' groups and the blocks they span, for a cluster of C CTAs
    auto split = [&](uint32_t C, uint32_t r) { return r >= C ? G : ((r * G) / C) & ~1u; };
    auto max_blocks = [&](uint32_t C) {
        uint32_t m = 0;
        for (uint32_t r = 0; r < C; ++r) {
            const uint32_t a = split(C, r), b = split(C, r + 1);
            if (b > a) m = std::max(m, (b - 1) / 8 - a / 8 + 1);
        }
        return m;
    };
    auto max_groups = [&](uint32_t C) {
        uint32_t m = 0;
        for (uint32_t r = 0; r < C; ++r) m = std::max(m, split(C, r + 1) - split(C, r));
        return m;
    };
    // the smallest cluster whose CTAs rotate their blocks in one round (pairs)
    uint32_t C = 1;
    while (C < 4 && (max_blocks(C) > kPairs || max_groups(C) > (uint32_t)kThreads)) C *= 2;
    uint64_t units = C == 1 ? (uint64_t)sms : (uint64_t)max_clusters(C, smem_limit, sms);
    uint64_t R = (g.n + units - 1) / units;
    if (C > 1 && R > kMaxClusterRows) {
        if (max_groups(1) > (uint32_t)kThreads) return false;
        C = 1;
        units = (uint64_t)sms;
        R = (g.n + units - 1) / units;
    }
    const bool cluster = C > 1;
    const uint32_t ng_max = max_groups(C);
    if (ng_max == 0 || ng_max > (uint32_t)kThreads) return false;
    const uint64_t used = (g.n + R - 1) / R;
    // high bytes and scales of a CTA's groups rounded out to 8 groups; a slot holds
    // the widest rank's
    uint32_t hb_max = 0;
    for (uint32_t r = 0; r < C; ++r) {
        const uint32_t a = split(C, r), b = split(C, r + 1);
        hb_max = std::max(hb_max, 2 * (((b + 7) & ~7u) - (a & ~7u)));
    }
    const uint32_t nsets = (uint32_t)kThreads / ng_max;
    const uint32_t u = nsets >= 32 ? 1 : 2;
    const uint32_t br = nsets * u;
    const uint64_t nbatch = (R + br - 1) / br;
    // base boxes of wg groups (3 wg <= 255 elements; even, so that every box starts 16-byte aligned)
    const uint32_t nbx = (ng_max + 83) / 84;
    const uint32_t wg = ((ng_max + nbx - 1) / nbx + 1) & ~1u;
    if (nbatch >= (1ull << 29) || hb_max / 8 > 256 || br > 256) return false;
    // a slot: the batch's base boxes, high bytes and scales, each box 128-byte aligned
    auto a128 = [](uint32_t b) { return (b + 127) / 128 * 128; };
    const uint32_t bstride = a128(br * 24 * wg);
    const uint32_t slot_high = nbx * bstride, slot_scale = slot_high + a128(br * hb_max);
    const uint32_t slot = slot_scale + a128(br * hb_max);
    const uint32_t part_stride = br | 1u;      // odd: the writers' lanes hit distinct banks
    const uint32_t part_slot = (ng_max * part_stride * 4 + 15) / 16 * 16;
    const uint32_t act = (ng_max * (kActGroupBytes + 8) + 15) / 16 * 16;
    // row sums (a whole number of 4-row vectors past R), then the inbox: C parts of
    // ceil(R / C) rows rounded up to a multiple of 4
    const uint64_t rq = ((R + C - 1) / C + 3) & ~3ull;
    const uint32_t rs_bytes = cluster ? (uint32_t)((((R + 3) & ~3ull) + C * rq) * 4) : 0u;
    const uint32_t bar_bytes = kBarBytes;
    const int64_t avail = (int64_t)smem_limit - kRegion0 - rs_bytes - bar_bytes;
    uint32_t nslots = (uint32_t)std::min<uint64_t>(kMaxSlots, nbatch);
    while (nslots > 0 && (int64_t)nslots * slot + std::max<int64_t>(act, (int64_t)nslots * part_slot) > avail)
        --nslots;
    if (nslots == 0 || (nslots < 2 && nbatch > 1) || slot >= (1u << 20)) return false;
    plan->ok = true;
    plan->cluster = C;
    plan->grid = (uint32_t)(C * used);
    plan->units = (uint32_t)used;
    plan->rows_per_cta = (uint32_t)R;
    plan->ng = ng_max;
    plan->hbytes = hb_max;
    plan->wg = wg;
    plan->nbx = nbx;
    plan->bstride = bstride;
    plan->nsets = nsets;
    plan->u = u;
    plan->nslots = nslots;
    plan->pre_issue = 1;
    plan->slot_bytes = slot;
    plan->slot_high = slot_high;
    plan->slot_scale = slot_scale;
    plan->part_stride = part_stride;
    plan->part_slot_bytes = part_slot;
    uint32_t off = kRegion0;      // the table (and, before it, the rotation scratch) starts the shared memory
    plan->off_ring = off;
    off += nslots * slot;
    plan->off_part = off;
    off += std::max(act, nslots * part_slot);
    plan->off_rs = off;
    off += rs_bytes;
    plan->off_bar = off;
    off += bar_bytes;
    plan->smem = off;
    plan->workspace = 0;
    return true;
}

int gemv_ptq1_int_launch(const Ptq1Plan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, void *workspace,
                         cudaStream_t stream, bool pdl) {
    (void)workspace;
    Ptq1Params p;
    std::memset(&p, 0, sizeof p);
    const uint8_t *base = payload + g.base_offset, *high = payload + g.high_offset, *scale = payload + g.scale_offset;
    if (!aligned(base, 16) || !aligned(high, 16) || !aligned(scale, 16))
        return fail(NINFER_ERR_ALIGNMENT, "ptq1 gemv: planes must start 16-byte aligned");
    const uint64_t G = g.groups_per_row, R = plan.rows_per_cta, U = plan.units, last_rows = g.n - (U - 1) * R;
    const uint32_t br = plan.nsets * plan.u;
    const uint32_t bbox[3] = {3 * plan.wg, br, 1}, hbox[3] = {plan.hbytes / 8, br, 1};
    int st = NINFER_OK;
    if (U > 1) {
        st = encode_3d_u64(&p.bmap_main, base, {3 * G, R, U - 1}, {g.base_row_bytes, R * g.base_row_bytes}, bbox);
        if (!st) st = encode_3d_u64(&p.hmap_main, high, {G / 4, R, U - 1}, {g.high_row_bytes, R * g.high_row_bytes}, hbox);
        if (!st)
            st = encode_3d_u64(&p.smap_main, scale, {G / 4, R, U - 1}, {g.scale_row_bytes, R * g.scale_row_bytes}, hbox);
        if (st) return st;
    }
    const uint64_t lr = (U - 1) * R;
    st = encode_3d_u64(&p.bmap_last, base + lr * g.base_row_bytes, {3 * G, last_rows, 1},
                       {g.base_row_bytes, last_rows * g.base_row_bytes}, bbox);
    if (!st)
        st = encode_3d_u64(&p.hmap_last, high + lr * g.high_row_bytes, {G / 4, last_rows, 1},
                           {g.high_row_bytes, last_rows * g.high_row_bytes}, hbox);
    if (!st)
        st = encode_3d_u64(&p.smap_last, scale + lr * g.scale_row_bytes, {G / 4, last_rows, 1},
                           {g.scale_row_bytes, last_rows * g.scale_row_bytes}, hbox);
    if (st) return st;
    p.x = x;
    p.signs = signs;
    p.y = y;
    p.n = g.n;
    p.units = plan.units;
    p.k = (uint32_t)g.k;
    p.groups = (uint32_t)g.groups_per_row;
    p.hbytes = plan.hbytes;
    p.rows_per_cta = plan.rows_per_cta;
    p.nsets = plan.nsets;
    p.u = plan.u;
    p.wg = plan.wg;
    p.nbx = plan.nbx;
    p.bstride = plan.bstride;
    p.nslots = plan.nslots;
    p.nslots_inv = (uint32_t)((1ull << 32) / plan.nslots + 1);
    p.pre_issue = pdl ? plan.pre_issue : 0u;
    p.slot_bytes = plan.slot_bytes;
    p.slot_high = plan.slot_high;
    p.slot_scale = plan.slot_scale;
    p.part_stride = plan.part_stride;
    p.part_slot_bytes = plan.part_slot_bytes;
    p.off_ring = plan.off_ring;
    p.off_part = plan.off_part;
    p.off_rs = plan.off_rs;
    p.off_bar = plan.off_bar;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.wait_cycles = wait_limit_cycles();
    st = device_error_word(&p.err);
    if (st) return st;
    void (*kernel)(Ptq1Params) =
        plan.u == 1 ? (x_dtype == NINFER_F32    ? gemv_ptq1_int_kernel<NINFER_F32, 1>
                       : x_dtype == NINFER_BF16 ? gemv_ptq1_int_kernel<NINFER_BF16, 1>
                                                : gemv_ptq1_int_kernel<NINFER_F16, 1>)
                    : (x_dtype == NINFER_F32    ? gemv_ptq1_int_kernel<NINFER_F32, 2>
                       : x_dtype == NINFER_BF16 ? gemv_ptq1_int_kernel<NINFER_BF16, 2>
                                                : gemv_ptq1_int_kernel<NINFER_F16, 2>);
    st = set_smem_attribute((const void *)kernel, (int)plan.smem);
    if (st) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = plan.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan.cluster > 1 ? 2 : 1;     // no cluster attribute at all unless clusters are wanted
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
