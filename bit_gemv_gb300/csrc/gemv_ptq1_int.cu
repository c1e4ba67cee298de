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
// Activation: warp pairs rotate and round it (rot2.cuh), write its 16-bit
// values in natural order to their scratch and pack, per group, 64 operand
// words: for base byte j (< 24), (x16[5j], x16[5j+1]) and (x16[5j+2],
// x16[5j+3]); for the four bytes 4q .. 4q+3, the pairs of their fifth weights
// (x16[5(4q+2c)+4], x16[5(4q+2c+1)+4]); for high byte h, its two pairs. With
// more than seven 1024-blocks, two CTAs of a cluster share the rotations and
// each writes its groups into both tables.
//
// Arithmetic: a 256-entry table maps a code byte to its digits as bytes
// (t0 | t1 << 8 | t2 << 16 | t3 << 24, with t4 in bits 2-3 of byte 0), held 32
// times so that lane l always reads bank l (entry B of lane l at B * 128 + 4 l,
// from the start of shared memory). Per base byte dp2a multiplies (t0, t1) and
// (t2, t3) by their activation pairs; the t4 fields of four consecutive bytes
// are gathered into one word by byte permutes and multiplied by their pairs
// (times 4, removed at the end); all exact in int32. Per group:
//   y += scale * 2^-E * (sum t x16 - sum x16)                    (value = t - 1)
//
// Work: one CTA per SM owns a contiguous range of rows, in tiles of 32 kRL
// rows (lane l: rows l, l + 32, .. of the tile, so that the 64 operand words of
// a group, read once into registers, serve kRL rows). A chunk of the ring is a
// tile's 16 groups: three 128-byte-swizzled boxes of base bytes (384 bytes per
// row), one box of high bytes and one of scales, on one mbarrier; warp w takes
// group w of the chunk, or half of group w % 8 when the chunk has only eight
// groups. With kRL = 1 a CTA whose rows exceed a multiple of 32 by one or two
// copies those rows whole into shared memory and computes them with lanes =
// (row, group). One chunk is requested before the programmatic-dependent-
// launch wait; the rest of the ring, by a warp that does not rotate, once x
// has arrived.
#include <cstring>

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

constexpr int kThreads = 512;
constexpr int kWarps = 16;
constexpr int kProducer = kWarps - 1;       // issues the ring; never rotates
constexpr uint32_t kChunkGroups = 16;
constexpr uint32_t kMaxSlots = 8;
constexpr uint32_t kMaxRem = 2;             // extra rows beyond whole 32-row tiles handled per (row, group)
constexpr uint32_t kActWords = 64;
// Groups sit kActStride words apart: the 4-word pad moves consecutive groups 16
// bytes along the banks, so the remainder-row path (lanes = 16 groups) reads
// its operand words with at most two-way conflicts; the tile path reads one
// group per warp (a broadcast) either way.
constexpr uint32_t kActStride = 68;
static_assert(kActStride >= kActWords && kActStride % 4 == 0, "operand words: 16-byte aligned groups");
constexpr uint32_t kActGroupBytes = kActStride * 4;
constexpr uint32_t kLutBytes = 256 * 128;   // entry B at B * 128: 32 lane copies
constexpr uint32_t kBarX = 1;               // named barrier: x has arrived
constexpr uint32_t kBarPair0 = 2;           // named barriers 2.. : one per rotating pair
constexpr uint32_t kMaxPairs = 7;           // warps 0-13
static_assert(kMaxPairs * kRotScratchBytes <= kLutBytes, "rotation scratch lives where the table is built later");

template <int kRL>
struct Tile {
    static constexpr uint32_t rows = 32 * kRL;
    static constexpr uint32_t base_box = 128 * rows;                   // one 128-byte column of base bytes
    static constexpr uint32_t chunk_bytes = 3 * base_box + 2 * 32 * rows;
};

struct Ptq1Params {
    CUtensorMap bmap_main, bmap_last;   // base rows {row bytes, R rows, CTA} / last CTA with rows, 128-byte boxes
    CUtensorMap hmap_main, hmap_last;   // high rows, 32-byte boxes
    CUtensorMap smap_main, smap_last;   // scale rows, 32-byte boxes
    const uint8_t *base, *high, *scale; // plane starts (remainder rows)
    uint64_t base_row, high_row, scale_row;
    const void *x;
    const uint16_t *signs;
    uint32_t act_bytes;
    void *y;
    uint64_t n;
    uint32_t k, groups, nblk, nch, rows_per_cta, grid_rows;     // nch: chunks per tile
    int x_dtype, y_dtype;
    uint32_t nslots, nslots_inv, pre_issue, nrot;               // nrot: rotating pairs at most
    uint32_t off_ring, off_act, off_rem, off_part, off_bar, off_cnt;     // table / rotation scratch at 0
    uint32_t *err;
    long long wait_cycles;
};

struct CtaRows {
    uint64_t begin;
    uint32_t ntile, rem;    // tiles (the last may be partial when rem == 0), remainder rows
    uint32_t rows;
};

template <int kRL>
__device__ __forceinline__ CtaRows cta_rows(const Ptq1Params &p) {
    CtaRows c;
    c.begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t end = c.begin + p.rows_per_cta < p.n ? c.begin + p.rows_per_cta : p.n;
    c.rows = end > c.begin ? (uint32_t)(end - c.begin) : 0u;
    const uint32_t T = Tile<kRL>::rows, full = c.rows / T, extra = c.rows % T;
    if (kRL == 1 && full >= 1 && extra <= kMaxRem) {
        c.ntile = full;
        c.rem = extra;
    } else {
        c.ntile = full + (extra ? 1 : 0);
        c.rem = 0;
    }
    return c;
}

// Chunk i = tile * nch + ch: its three base boxes, high box and scale box into ring slot i % nslots.
template <int kRL>
__device__ __forceinline__ void issue_chunk(const Ptq1Params &p, uint8_t *smem, uint32_t item, bool last_cta) {
    using T = Tile<kRL>;
    const uint32_t tile = item / p.nch, ch = item % p.nch, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * T::chunk_bytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, T::chunk_bytes);
    const int y0 = (int)(tile * T::rows), z = (int)blockIdx.x;
#pragma unroll
    for (int bx = 0; bx < 3; ++bx) {
        const int x = (int)(ch * 384 + 128 * bx);
        if (last_cta) tma_load_2d(dst + bx * T::base_box, &p.bmap_last, x, y0, bar);
        else tma_load_3d(dst + bx * T::base_box, &p.bmap_main, x, y0, z, bar);
    }
    const int xh = (int)(ch * 32);
    if (last_cta) {
        tma_load_2d(dst + 3 * T::base_box, &p.hmap_last, xh, y0, bar);
        tma_load_2d(dst + 3 * T::base_box + 32 * T::rows, &p.smap_last, xh, y0, bar);
    } else {
        tma_load_3d(dst + 3 * T::base_box, &p.hmap_main, xh, y0, z, bar);
        tma_load_3d(dst + 3 * T::base_box + 32 * T::rows, &p.smap_main, xh, y0, z, bar);
    }
}

// Rotates block b with the pair and writes the operand words and group entries
// {2^-E (with the transform's 1/32), sum of the group's x16 (int bits)} of its
// eight groups into act and, when act_remote is non-zero (the cluster address
// of the same table in the other CTA of the cluster), into that table too.
__device__ __forceinline__ void rotate_pack_ptq1(bool rotate, float (&v)[16], const float (&d)[16], uint32_t b,
                                                 uint32_t groups, uint8_t *act, uint32_t act_remote, float *scr,
                                                 int t, uint32_t bar) {
    const int lane = t & 31;
    uint32_t qb[16];
    const int E = rotate_quant2(rotate, v, d, scr, t, bar, qb);
    const float f = ldexpf(1.f, -E - (rotate ? 5 : 0));
    // x16 in natural order (int16) in the scratch: elements 512 i + 8 t .. + 7
    int16_t *qs = reinterpret_cast<int16_t *>(scr);
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
        const uint32_t G = b * 8 + 4 * i + (t >> 4);
        if ((lane & 15) == 0 && G < groups) {
            const int sg = lane < 16 ? s_lo : s_hi;
            reinterpret_cast<float2 *>(act + (uint64_t)groups * kActGroupBytes)[G] = make_float2(f, __int_as_float(sg));
            if (act_remote) st_cluster_v2(act_remote + groups * kActGroupBytes + 8 * G, __float_as_uint(f), (uint32_t)sg);
        }
    }
    named_barrier(bar, 64);
    // operand words: the block's 8 groups have 208 code bytes (192 base, 16 high);
    // thread t takes bytes t, t + 64, t + 128 and t + 192
    uint32_t *aw = reinterpret_cast<uint32_t *>(act);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = t + 64 * i;
        if (u >= 208) break;
        const uint32_t gl = u < 192 ? u / 24 : (u - 192) >> 1, G = b * 8 + gl;
        if (G >= groups) continue;
        uint32_t *dst = aw + (uint64_t)G * kActStride;
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
    named_barrier(bar, 64);
    if (act_remote) {
        // the block's groups as they now stand in this table, to the other CTA of the cluster
        const uint32_t g0 = b * 8, ng = g0 + 8 <= groups ? 8 : (g0 < groups ? groups - g0 : 0);
        const uint32_t n16 = ng * kActGroupBytes / 16;
        const uint4 *src = reinterpret_cast<const uint4 *>(act + (uint64_t)g0 * kActGroupBytes);
        for (uint32_t c = t; c < n16; c += 64) st_cluster_v4(act_remote + g0 * kActGroupBytes + 16 * c, src[c]);
    }
    named_barrier(bar, 64);      // the scratch may be reused
}

// sum_j t_j x16_j over kNq base words (four code bytes each) and kNh high
// bytes of one group (a whole group: 6 and 2; half a group: 3 and 1), from the
// operand words av (in registers, in the order of the group's 64 words: the
// pairs of base byte j at 2 j, the fifth-weight pairs of word q at kT4 + 2 q,
// the pairs of high byte h at kHi + 2 h) and the lane's copies of the digit
// table: entry B of this lane at lut + (B << 7 | lane4), lane4 = 4 * lane.
template <int kNq, int kNh, int kT4, int kHi, int kN>
__device__ __forceinline__ int group_dot(const uint32_t (&bw)[kNq], uint32_t hb, uint32_t lut, uint32_t lane4,
                                         const uint32_t (&av)[kN]) {
    int acc[4] = {0, 0, 0, 0}, acc4 = 0;
#pragma unroll
    for (int q = 0; q < kNq; ++q) {
        uint32_t W[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int sh = 8 * c - 7;
            const uint32_t off = ((sh >= 0 ? bw[q] >> sh : bw[q] << (-sh)) & 0x7F80u) | lane4;
            W[c] = lds32(lut + off);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t m = W[c] & 0x03030303u;
            const int j = 4 * q + c;
            acc[c] = dp2a_lo(av[2 * j], m, acc[c]);
            acc[c] = dp2a_hi(av[2 * j + 1], m, acc[c]);
        }
        // byte 0 of each entry holds 4 * t4 in bits 2-3: gather the four
        const uint32_t g = __byte_perm(__byte_perm(W[0], W[1], 0x0040u), __byte_perm(W[2], W[3], 0x0040u), 0x5410u) &
                           0x0C0C0C0Cu;
        acc4 = dp2a_lo(av[kT4 + 2 * q], g, acc4);
        acc4 = dp2a_hi(av[kT4 + 2 * q + 1], g, acc4);
    }
#pragma unroll
    for (int hh = 0; hh < kNh; ++hh) {
        const int sh = 8 * hh - 7;
        const uint32_t off = ((sh >= 0 ? hb >> sh : hb << (-sh)) & 0x7F80u) | lane4;
        const uint32_t m = lds32(lut + off) & 0x03030303u;
        acc[hh] = dp2a_lo(av[kHi + 2 * hh], m, acc[hh]);
        acc[hh] = dp2a_hi(av[kHi + 2 * hh + 1], m, acc[hh]);
    }
    return acc[0] + acc[1] + acc[2] + acc[3] + (acc4 >> 2);
}

template <int kN>
__device__ __forceinline__ void load_words(const uint32_t *src, uint32_t (&av)[kN]) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < kN / 4; ++i) {
        const uint4 a = s4[i];
        av[4 * i] = a.x;
        av[4 * i + 1] = a.y;
        av[4 * i + 2] = a.z;
        av[4 * i + 3] = a.w;
    }
}

template <int kRL, int kXType>
__global__ void __launch_bounds__(kThreads, 1) gemv_ptq1_int_kernel(const __grid_constant__ Ptq1Params p) {
    using TL = Tile<kRL>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const CtaRows cr = cta_rows<kRL>(p);
    const bool last_cta = blockIdx.x == p.grid_rows - 1;
    const uint32_t nitems = cr.ntile * p.nch;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t rem_bar = bar0 + 8 * kMaxSlots;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1;
    const uint32_t lut_s = smem_u32(smem), lane4 = 4u * (uint32_t)lane;
    uint8_t *rem_s = smem + p.off_rem;
    uint8_t *act_s = smem + p.off_act;
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    const uint32_t pre = p.pre_issue < ring_to ? p.pre_issue : ring_to;
    // rotation tasks = 1024-blocks; in a cluster of two CTAs each takes every
    // other block (local task i is block 2 i + rank) and writes both tables
    const uint32_t csize = cluster_nctarank(), crank = cluster_ctarank();
    const uint32_t ntask = csize == 2 ? (p.nblk + 1 - crank) / 2 : p.nblk;
    auto task_of = [&](uint32_t i) { return csize == 2 ? 2 * i + crank : i; };
    const uint32_t npr = ntask < p.nrot ? ntask : p.nrot;
    const uint32_t pr = (uint32_t)warp >> 1;
    const int t = tid & 63;
    const bool rotating = pr < npr;
    const uint32_t nwait = 32 * (2 * npr + 1);
    const uint32_t act_remote0 = csize == 2 ? mapa_shared(smem_u32(act_s), crank ^ 1u) : 0u;

    if (tid == kProducer * 32) {
        prefetch_tmap(last_cta ? &p.bmap_last : &p.bmap_main);
        prefetch_tmap(last_cta ? &p.hmap_last : &p.hmap_main);
        prefetch_tmap(last_cta ? &p.smap_last : &p.smap_main);
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        mbar_init(rem_bar, 1);
        *failed = 0;
        fence_mbar_init();
        // weights are read-only parameters: the first chunks and the remainder rows before the dependency wait
        for (uint32_t i = 0; i < pre; ++i) issue_chunk<kRL>(p, smem, i, last_cta);
        *issued = pre;
        if (cr.rem) {
            const uint32_t rb_bytes = (uint32_t)(p.base_row + p.high_row + p.scale_row);
            mbar_arrive_expect_tx(rem_bar, cr.rem * rb_bytes);
            for (uint32_t rr = 0; rr < cr.rem; ++rr) {
                const uint64_t r = cr.begin + (uint64_t)cr.ntile * TL::rows + rr;
                const uint32_t dd = smem_u32(rem_s) + rr * rb_bytes;
                bulk_g2s(dd, p.base + r * p.base_row, (uint32_t)p.base_row, rem_bar);
                bulk_g2s(dd + (uint32_t)p.base_row, p.high + r * p.high_row, (uint32_t)p.high_row, rem_bar);
                bulk_g2s(dd + (uint32_t)(p.base_row + p.high_row), p.scale + r * p.scale_row, (uint32_t)p.scale_row,
                         rem_bar);
            }
        }
    }
    float v[16], d[16];
    if (rotating) {
        // the first rotation of a rotating pair
        const uint32_t b = task_of(pr);
        float *scr = reinterpret_cast<float *>(smem + pr * kRotScratchBytes);
        if (p.signs) load_signs2(p.signs, b, t, d);     // read-only
        pdl_launch_dependents();
        pdl_wait();          // x may come from the preceding kernel
        load_block2<kXType>(p.x, p.k, b, t, v);
        // x has arrived once its first and last values can be stored; then the
        // producer may queue the rest of the ring behind it
        *reinterpret_cast<volatile float *>(scr + 1080 + (t >> 5)) = v[0] + v[15];
        named_barrier_arrive(kBarX, nwait);
        rotate_pack_ptq1(p.signs != nullptr, v, d, b, p.groups, act_s, act_remote0, scr, t, kBarPair0 + pr);
    } else {
        pdl_launch_dependents();
        pdl_wait();
        if (warp == kProducer) {
            // the rest of the ring, once x has arrived in every rotating warp
            named_barrier(kBarX, nwait);
            if (lane == 0) {
                for (uint32_t i = pre; i < ring_to; ++i) issue_chunk<kRL>(p, smem, i, last_cta);
                *issued = ring_to;
            }
            __syncwarp();
        }
    }
#pragma unroll 1
    for (uint32_t i = pr + npr; rotating && i < ntask; i += npr) {     // more blocks than rotating pairs
        const uint32_t b = task_of(i);
        if (p.signs) load_signs2(p.signs, b, t, d);
        load_block2<kXType>(p.x, p.k, b, t, v);
        rotate_pack_ptq1(p.signs != nullptr, v, d, b, p.groups, act_s, act_remote0,
                         reinterpret_cast<float *>(smem + pr * kRotScratchBytes), t, kBarPair0 + pr);
    }
    // the operand words are complete in both CTAs of a cluster; the rotation
    // scratch is free for the digit table
    if (csize == 2) cluster_sync();
    else __syncthreads();
    {
        // digit table, replicated per bank: entry (B, l) at word 32 B + l; thread
        // tid computes entry tid / 2 and writes 16 of its copies
        uint32_t B = (uint32_t)tid >> 1, W = 0;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint32_t dg = B % 3;
            B /= 3;
            W |= i < 4 ? dg << (8 * i) : dg << 2;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(smem + ((tid >> 1) * 32 + 16 * (tid & 1)) * 4);
        const uint4 w4 = make_uint4(W, W, W, W);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = w4;
    }
    __syncthreads();

    bool ok = true;
    const uint32_t *act_w = reinterpret_cast<const uint32_t *>(act_s);
    const float2 *gs = reinterpret_cast<const float2 *>(act_s + (uint64_t)p.groups * kActGroupBytes);
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    float *part_rem = part + kWarps * TL::rows;      // [kMaxRem][groups]

    // remainder rows: lanes = (row, group of the chunk); warp w takes chunks w, w + 16, ...
    if (cr.rem) {
        ok = ok && mbar_wait(rem_bar, 0, p.err, p.wait_cycles);
        const uint32_t rb_bytes = (uint32_t)(p.base_row + p.high_row + p.scale_row);
        const uint32_t rr = lane >> 4;
        for (uint32_t ch = warp; ok && ch < p.nch; ch += kWarps) {
            const uint32_t G = ch * kChunkGroups + (lane & 15);
            if (rr < cr.rem && G < p.groups) {
                const uint8_t *row = rem_s + rr * rb_bytes;
                const uint2 q0 = *reinterpret_cast<const uint2 *>(row + 24 * G);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(row + 24 * G + 8);
                const uint2 q2 = *reinterpret_cast<const uint2 *>(row + 24 * G + 16);
                const uint32_t bw[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
                const uint32_t hb = *reinterpret_cast<const uint16_t *>(row + p.base_row + 2 * G);
                const float s = __half2float(*reinterpret_cast<const __half *>(row + p.base_row + p.high_row + 2 * G));
                const float2 f = gs[G];
                uint32_t av[64];
                load_words(act_w + G * kActStride, av);
                const int dot = group_dot<6, 2, 48, 60>(bw, hb, lut_s, lane4, av);
                part_rem[rr * p.groups + G] = s * f.x * (float)(dot - __float_as_int(f.y));
            }
        }
    }

    // tiles: warp w takes group 16 ch + w of chunk (tile, ch), or half of group
    // 16 ch + w % 8 when the chunk has eight groups; lane l: rows l + 32 q
    // the 24 base bytes of group g of a chunk's row: three 8-byte words in the
    // swizzled 128-byte columns (row % 8 pattern); g = warp for a whole group,
    // warp % 8 for half a group
    auto base_off = [&](uint32_t g, int i) {
        const uint32_t o = 24 * g + 8 * i, bx = o >> 7, c16 = (o & 127) >> 4, hf = (o >> 3) & 1;
        return bx * TL::base_box + lane * 128 + ((c16 ^ (lane & 7)) << 4) + 8 * hf;
    };
    const uint32_t bo_f0 = base_off(warp, 0), bo_f1 = base_off(warp, 1), bo_f2 = base_off(warp, 2);
    const uint32_t bo_h0 = base_off(warp & 7, 0), bo_h1 = base_off(warp & 7, 1), bo_h2 = base_off(warp & 7, 2);
#pragma unroll 1
    for (uint32_t tile = 0; tile < cr.ntile; ++tile) {
        float y[kRL];
#pragma unroll
        for (int q = 0; q < kRL; ++q) y[q] = 0.f;
#pragma unroll 1
        for (uint32_t ch = 0; ch < p.nch; ++ch) {
            const uint32_t item = tile * p.nch + ch;
            const uint32_t cycle = __umulhi(item, p.nslots_inv);      // item / nslots (item < 2^29)
            const uint32_t slot = item - cycle * p.nslots, phase = cycle & 1;
            const bool half = p.groups - ch * kChunkGroups <= 8;       // a chunk of eight groups
            const uint32_t gw = half ? (uint32_t)(warp & 7) : (uint32_t)warp, hh = half ? (uint32_t)(warp >> 3) : 0u;
            const uint32_t G = ch * kChunkGroups + gw;
            ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err, p.wait_cycles);
            if (ok && G < p.groups) {
                const uint8_t *sa = smem + p.off_ring + slot * TL::chunk_bytes;
                const float2 f = gs[G];
                if (!half) {
                    uint32_t av[64];
                    load_words(act_w + G * kActStride, av);
                    const int off = __float_as_int(f.y);
#pragma unroll
                    for (int q = 0; q < kRL; ++q) {
                        const uint32_t ro = q * 32 * 128;      // row lane + 32 q of each base box
                        const uint2 b0 = *reinterpret_cast<const uint2 *>(sa + bo_f0 + ro);
                        const uint2 b1 = *reinterpret_cast<const uint2 *>(sa + bo_f1 + ro);
                        const uint2 b2 = *reinterpret_cast<const uint2 *>(sa + bo_f2 + ro);
                        const uint32_t bw[6] = {b0.x, b0.y, b1.x, b1.y, b2.x, b2.y};
                        const uint32_t r = lane + 32 * q;
                        const uint32_t hb = *reinterpret_cast<const uint16_t *>(sa + 3 * TL::base_box + r * 32 + 2 * gw);
                        const float s = __half2float(
                            *reinterpret_cast<const __half *>(sa + 3 * TL::base_box + 32 * TL::rows + r * 32 + 2 * gw));
                        const int dot = group_dot<6, 2, 48, 60>(bw, hb, lut_s, lane4, av);
                        y[q] = fmaf(s * f.x, (float)(dot - off), y[q]);
                    }
                } else {
                    // half hh of the group: base words 3 hh .. 3 hh + 2 (bytes 12 hh .. 12 hh + 11),
                    // high byte hh; its 32 operand words: base pairs 24 hh .., fifth-weight
                    // pairs 48 + 6 hh .., high pairs 60 + 2 hh ..
                    const uint32_t *src = act_w + G * kActStride;
                    uint32_t avh[32];
                    load_words<24>(src + 24 * hh, *reinterpret_cast<uint32_t(*)[24]>(avh));
                    // (8-byte aligned: a group starts 16-byte aligned, word 48 + 6 hh at byte 192 + 24 hh)
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        const uint2 t4 = *reinterpret_cast<const uint2 *>(src + 48 + 6 * hh + 2 * i);
                        avh[24 + 2 * i] = t4.x;
                        avh[25 + 2 * i] = t4.y;
                    }
                    const uint2 hi = *reinterpret_cast<const uint2 *>(src + 60 + 2 * hh);
                    avh[30] = hi.x; avh[31] = hi.y;
                    const int off = hh ? 0 : __float_as_int(f.y);
#pragma unroll
                    for (int q = 0; q < kRL; ++q) {
                        const uint32_t ro = q * 32 * 128;
                        const uint2 b0 = *reinterpret_cast<const uint2 *>(sa + bo_h0 + ro);
                        const uint2 b1 = *reinterpret_cast<const uint2 *>(sa + bo_h1 + ro);
                        const uint2 b2 = *reinterpret_cast<const uint2 *>(sa + bo_h2 + ro);
                        const uint32_t bh[3] = {hh ? b1.y : b0.x, hh ? b2.x : b0.y, hh ? b2.y : b1.x};
                        const uint32_t r = lane + 32 * q;
                        const uint32_t hb = *reinterpret_cast<const uint16_t *>(sa + 3 * TL::base_box + r * 32 + 2 * gw);
                        const float s = __half2float(
                            *reinterpret_cast<const __half *>(sa + 3 * TL::base_box + 32 * TL::rows + r * 32 + 2 * gw));
                        const int dot = group_dot<3, 1, 24, 30>(bh, hh ? hb >> 8 : hb, lut_s, lane4, avh);
                        y[q] = fmaf(s * f.x, (float)(dot - off), y[q]);
                    }
                }
            }
            // release the slot; the last of its sixteen readers refills it with the chunk nslots further on
            __syncwarp();
            if (lane == 0) {
                if (!ok) *failed = 1;
                __threadfence_block();
                const uint32_t seen = atomicAdd(&cnt[slot], 1u);
                if (seen == kWarps - 1) {
                    cnt[slot] = 0;
                    if (ok && !*(volatile uint32_t *)failed && item + p.nslots < nitems) {
                        fence_proxy_async();
                        issue_chunk<kRL>(p, smem, item + p.nslots, last_cta);
                        atomicAdd(issued, 1u);
                    }
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int q = 0; q < kRL; ++q) part[warp * TL::rows + 32 * q + lane] = y[q];
        __syncthreads();
        if (warp < kRL) {
            const uint32_t rl = warp * 32 + lane;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += part[w * TL::rows + rl];
            const uint32_t row = tile * TL::rows + rl;
            if (row < cr.rows - cr.rem) store1(p.y, cr.begin + row, p.y_dtype, acc);
        }
        __syncthreads();
    }
    if (cr.rem) {
        __syncthreads();       // part_rem complete (also when the CTA has no tile)
        if (warp == 0 && lane < cr.rem) {
            float acc = 0.f;
            for (uint32_t G = 0; G < p.groups; ++G) acc += part_rem[lane * p.groups + G];
            store1(p.y, cr.begin + (uint64_t)cr.ntile * TL::rows + lane, p.y_dtype, acc);
        }
    }
    // after a timed-out wait: let the copies still in flight land (at most one
    // per slot, the last one issued into it) before the CTA's memory is freed
    if (tid == 0 && *(volatile uint32_t *)failed) {
        const uint32_t n_issued = *(volatile uint32_t *)issued;
        for (uint32_t i = n_issued > p.nslots ? n_issued - p.nslots : 0; i < n_issued; ++i)
            mbar_wait(bar0 + 8 * (i % p.nslots), (i / p.nslots) & 1, p.err, 200000000ll);
        if (cr.rem) mbar_wait(rem_bar, 0, p.err, 200000000ll);
    }
}

}  // namespace

bool gemv_ptq1_int_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                        Ptq1Plan *plan) {
    *plan = Ptq1Plan{};
    if (M != 1) return false;
    if (rotate && g.k % 1024) return false;
    // high and scale rows must be whole 16-byte units (8 groups) for the boxes and bulk copies
    if (g.groups_per_row % 8 || g.base_row_bytes % 16 || g.high_row_bytes % 16 || g.scale_row_bytes % 16) return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31)) return false;
    const uint32_t groups = (uint32_t)g.groups_per_row;
    const uint32_t nblk = (uint32_t)((g.k + 1023) / 1024);
    const uint32_t nch = (groups + kChunkGroups - 1) / kChunkGroups;
    // one CTA per SM with ~n / SMs rows each; four rows per lane when a CTA has
    // 256 rows or more (the operand words of a group then serve four rows)
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)sms, g.n / 32));
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid_rows = (g.n + R - 1) / R;
    const int rl = R >= 256 ? 4 : 1;
    if ((uint64_t)nch * ((R + 32 * rl - 1) / (32 * rl)) >= (1ull << 29)) return false;
    // more blocks than rotating pairs: CTA pairs form clusters that share the rotations
    const bool cluster = grid_rows >= 2 && nblk > kMaxPairs;
    const uint64_t grid = cluster ? (grid_rows + 1) / 2 * 2 : grid_rows;
    const uint32_t ntask = cluster ? (nblk + 1) / 2 : nblk;
    const uint32_t nrot = std::min<uint32_t>(ntask, kMaxPairs);
    const uint32_t chunk = rl == 4 ? Tile<4>::chunk_bytes : Tile<1>::chunk_bytes;
    const uint32_t act_bytes = ((groups * (kActGroupBytes + 8) + 15) / 16) * 16;
    const uint32_t rem_bytes = rl == 1 ? (uint32_t)(kMaxRem * (g.base_row_bytes + g.high_row_bytes + g.scale_row_bytes)) : 0u;
    const uint32_t part_bytes = (kWarps * 32 * rl + (rl == 1 ? kMaxRem * groups : 0)) * 4;
    const uint32_t bar_bytes = (kMaxSlots + 2) * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 4) * 4;
    const uint32_t fixed = kLutBytes + act_bytes + ((rem_bytes + 15) / 16) * 16 + ((part_bytes + 15) / 16) * 16 +
                           bar_bytes + cnt_bytes;
    if ((int64_t)fixed + 2 * (int64_t)chunk > smem_limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((smem_limit - (int)fixed) / (int)chunk));
    plan->ok = true;
    plan->rl = rl;
    plan->cluster = cluster;
    plan->grid = (uint32_t)grid;
    plan->grid_rows = (uint32_t)grid_rows;
    plan->rows_per_cta = (uint32_t)R;
    plan->nch = nch;
    plan->nslots = nslots;
    plan->pre_issue = std::min<uint32_t>(1, nslots);
    plan->nrot = nrot;
    uint32_t off = kLutBytes;     // the table (and, before it, the rotation scratch) starts the shared memory
    plan->off_ring = off;
    off += nslots * chunk;
    plan->off_act = off;
    off += act_bytes;
    plan->off_rem = off;
    off += ((rem_bytes + 15) / 16) * 16;
    plan->off_part = off;
    off += ((part_bytes + 15) / 16) * 16;
    plan->off_bar = off;
    off += bar_bytes;
    plan->off_cnt = off;
    off += cnt_bytes;
    plan->smem = off;
    plan->act_bytes = act_bytes;
    plan->workspace = 0;
    return true;
}

int gemv_ptq1_int_launch(const Ptq1Plan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, void *workspace,
                         cudaStream_t stream, bool pdl) {
    (void)workspace;
    Ptq1Params p;
    std::memset(&p, 0, sizeof p);
    p.base = payload + g.base_offset;
    p.high = payload + g.high_offset;
    p.scale = payload + g.scale_offset;
    p.base_row = g.base_row_bytes;
    p.high_row = g.high_row_bytes;
    p.scale_row = g.scale_row_bytes;
    p.x = x;
    p.signs = signs;
    p.act_bytes = plan.act_bytes;
    p.y = y;
    p.n = g.n;
    p.k = (uint32_t)g.k;
    p.groups = (uint32_t)g.groups_per_row;
    p.nblk = (uint32_t)((g.k + 1023) / 1024);
    p.nch = plan.nch;
    p.rows_per_cta = plan.rows_per_cta;
    p.grid_rows = plan.grid_rows;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.nslots_inv = (uint32_t)((1ull << 32) / plan.nslots + 1);
    p.pre_issue = plan.pre_issue;
    p.nrot = plan.nrot;
    p.off_ring = plan.off_ring;
    p.off_act = plan.off_act;
    p.off_rem = plan.off_rem;
    p.off_part = plan.off_part;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    p.wait_cycles = wait_limit_cycles();
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint32_t box_rows = 32u * (uint32_t)plan.rl;
    const uint64_t R = plan.rows_per_cta, G = plan.grid_rows, last_rows = g.n - (G - 1) * R;
    if (G > 1) {
        st = encode_row_tiles(&p.bmap_main, p.base, g.base_row_bytes, R, G - 1, 128, box_rows, true);
        if (!st) st = encode_row_tiles(&p.hmap_main, p.high, g.high_row_bytes, R, G - 1, 32, box_rows, false);
        if (!st) st = encode_row_tiles(&p.smap_main, p.scale, g.scale_row_bytes, R, G - 1, 32, box_rows, false);
        if (st) return st;
    }
    const uint64_t lr = (G - 1) * R;
    st = encode_rows(&p.bmap_last, p.base + lr * g.base_row_bytes, g.base_row_bytes, last_rows, 128, box_rows, true);
    if (!st)
        st = encode_rows(&p.hmap_last, p.high + lr * g.high_row_bytes, g.high_row_bytes, last_rows, 32, box_rows,
                         false);
    if (!st)
        st = encode_rows(&p.smap_last, p.scale + lr * g.scale_row_bytes, g.scale_row_bytes, last_rows, 32, box_rows,
                         false);
    if (st) return st;
    void (*kernel)(Ptq1Params) = nullptr;
    if (plan.rl == 4) {
        kernel = x_dtype == NINFER_F32 ? gemv_ptq1_int_kernel<4, NINFER_F32>
                 : x_dtype == NINFER_BF16 ? gemv_ptq1_int_kernel<4, NINFER_BF16>
                                          : gemv_ptq1_int_kernel<4, NINFER_F16>;
    } else {
        kernel = x_dtype == NINFER_F32 ? gemv_ptq1_int_kernel<1, NINFER_F32>
                 : x_dtype == NINFER_BF16 ? gemv_ptq1_int_kernel<1, NINFER_BF16>
                                          : gemv_ptq1_int_kernel<1, NINFER_F16>;
    }
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
    attr[1].val.clusterDim.x = plan.cluster ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan.cluster ? 2 : 1;     // no cluster attribute at all unless CTA pairs are wanted
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
