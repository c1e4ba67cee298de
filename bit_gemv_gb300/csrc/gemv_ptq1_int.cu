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
// Arithmetic: the rotated activation is 16-bit fixed point per 1024-block
// (act16.cuh). A 256-entry table maps a code byte to its digits as bytes
// (t0 | t1 << 8 | t2 << 16 | t3 << 24, with t4 in bits 2-3 of byte 0); the
// table is replicated 32 times so that lane l always reads bank l (entry B of
// lane l at B * 128 + 4 l, from the start of shared memory). Per base byte,
// dp2a multiplies (t0, t1) and
// (t2, t3) by int16 activation pairs; the t4 fields of four consecutive bytes
// are gathered into one word by byte permutes and multiplied by two pairs of
// fifth activations (times 4, removed at the end), all exactly in int32. Per
// group:
//   y += scale * 2^-E * (sum t x16 - sum x16)                    (value = t - 1)
//
// Data movement: one CTA per SM owns a contiguous range of rows, processed as
// row blocks of 32 (lane = row, so each activation word read from shared
// memory is a broadcast). Items are 32 rows x 16 groups: three 128-byte-
// swizzled tensor boxes of base bytes (16 groups = 384 bytes per row), one box
// of high bytes and one of scales, on one mbarrier; warp w takes group w of
// each item. When a CTA's rows exceed a multiple of 32 by one or two, those
// rows are copied whole into shared memory (bulk copies issued before the
// dependency wait) and computed with lanes = (row, group). A few items are
// requested before the programmatic-dependent-launch wait; x is requested
// right after it and the rest of the ring behind it.
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

constexpr int kThreads = 512;     // 16 warps, one per group of an item; one CTA per SM
constexpr int kWarps = 16;
constexpr int kRows = 32;         // rows per block, one per lane
constexpr uint32_t kChunk = 16;   // groups per item
constexpr uint32_t kBaseBox = 128 * kRows;                 // 128 bytes of 32 rows
constexpr uint32_t kItemBytes = 3 * kBaseBox + 2 * 32 * kRows;
constexpr uint32_t kMaxSlots = 12;
constexpr uint32_t kRotPairs = 8;
constexpr uint32_t kMaxRem = 2;   // extra rows beyond whole row blocks handled per (row, group)
constexpr uint32_t kActWords = 64; // per group: 24 base bytes x 2 words + 6 t4 quads x 2 words + 2 high bytes x 2 words
// Groups sit kActStride words apart: the 4-word pad moves consecutive groups 16
// bytes along the banks, so the remainder-row path (lanes = 16 groups) reads
// its operand words with at most two-way conflicts; the row-block path reads
// one group per warp (a broadcast) either way.
constexpr uint32_t kActStride = 68;
static_assert(kActStride >= kActWords && kActStride % 4 == 0, "operand words: 16-byte aligned groups");
constexpr uint32_t kLutBytes = 256 * 128; // entry B at B * 128: 32 lane copies

struct Ptq1Params {
    CUtensorMap bmap_main, bmap_last;   // base rows {row bytes, R rows, CTA} / last CTA, boxes 128 B x 32 rows
    CUtensorMap hmap_main, hmap_last;   // high rows, boxes 32 B x 32 rows
    CUtensorMap smap_main, smap_last;   // scale rows, boxes 32 B x 32 rows
    const uint8_t *base, *high, *scale; // plane starts (remainder rows)
    uint64_t base_row, high_row, scale_row;
    const void *x;
    const uint16_t *signs;
    const uint8_t *act_g;               // operand words from ptq1_prep_kernel, or null (rotate here)
    uint32_t act_bytes;
    void *y;
    uint64_t n;
    uint32_t k, groups, nblk, nch, rows_per_cta;
    int x_dtype, y_dtype;
    uint32_t nslots, pre_issue;
    uint32_t off_ring, off_act, off_rot, off_rem, off_part, off_bar, off_cnt;     // the table is at offset 0
    uint32_t *err;
};

struct CtaRows {
    uint64_t begin;
    uint32_t nrb, rem;      // row blocks of 32 (the last may be partial when rem == 0), remainder rows
    uint32_t rows;
};

__device__ __forceinline__ CtaRows cta_rows(const Ptq1Params &p) {
    CtaRows c;
    c.begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t end = c.begin + p.rows_per_cta < p.n ? c.begin + p.rows_per_cta : p.n;
    c.rows = (uint32_t)(end - c.begin);
    const uint32_t full = c.rows / kRows, extra = c.rows % kRows;
    if (full >= 1 && extra <= kMaxRem) {
        c.nrb = full;
        c.rem = extra;
    } else {
        c.nrb = full + (extra ? 1 : 0);
        c.rem = 0;
    }
    return c;
}

// Item i = rb * nch + ch: its three base boxes, high box and scale box into ring slot i % nslots.
__device__ __forceinline__ void issue_item(const Ptq1Params &p, uint8_t *smem, uint32_t item, bool last_cta) {
    const uint32_t rb = item / p.nch, ch = item % p.nch, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kItemBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kItemBytes);
    const int y0 = (int)(rb * kRows), z = (int)blockIdx.x;
#pragma unroll
    for (int bx = 0; bx < 3; ++bx) {
        const int x = (int)(ch * 384 + 128 * bx);
        if (last_cta) tma_load_2d(dst + bx * kBaseBox, &p.bmap_last, x, y0, bar);
        else tma_load_3d(dst + bx * kBaseBox, &p.bmap_main, x, y0, z, bar);
    }
    const int xh = (int)(ch * 32);
    if (last_cta) {
        tma_load_2d(dst + 3 * kBaseBox, &p.hmap_last, xh, y0, bar);
        tma_load_2d(dst + 3 * kBaseBox + 32 * kRows, &p.smap_last, xh, y0, bar);
    } else {
        tma_load_3d(dst + 3 * kBaseBox, &p.hmap_main, xh, y0, z, bar);
        tma_load_3d(dst + 3 * kBaseBox + 32 * kRows, &p.smap_main, xh, y0, z, bar);
    }
}

// Operand words of block b from its x16 (rotate_quantize16): per group G,
//   word 2j + c (j < 24): c = 0 -> (x16[5j], x16[5j+1]), 1 -> (x16[5j+2], x16[5j+3])
//   word 48 + 2q + c (q < 6): (x16[5(4q+2c)+4], x16[5(4q+2c+1)+4])   (the t4 weights of bytes 4q .. 4q+3)
//   word 60 + 2h + c (h < 2): (x16[120+4h+2c], x16[121+4h+2c])
// and gs[G] = {2^-E, sum of the group's x16 (as int bits)}. The block's 8
// groups have 208 code bytes (192 base, 16 high); thread t of the pair takes
// bytes t, t + 64, t + 128 and t + 192.
__device__ __forceinline__ void pack_ptq1(const int16_t *qs, uint8_t *act_s, uint32_t groups, uint32_t b, int t, int E,
                                          uint32_t bar) {
    uint32_t *act = reinterpret_cast<uint32_t *>(act_s);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = t + 64 * i;
        if (u >= 208) break;
        const uint32_t gl = u < 192 ? u / 24 : (u - 192) >> 1, G = b * 8 + gl;
        if (G >= groups) continue;
        uint32_t *dst = act + (uint64_t)G * kActStride;
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
    // group sums: thread t sums elements 16t .. 16t + 15 (group t / 8)
    int sum = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) sum += qs[16 * t + e];
#pragma unroll
    for (int sh = 4; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
    const uint32_t G = b * 8 + (t >> 3);
    if ((t & 7) == 0 && G < groups)
        reinterpret_cast<float2 *>(act_s + (uint64_t)groups * kActStride * 4)[G] =
            make_float2(ldexpf(1.f, -E), __int_as_float(sum));
    named_barrier(bar, 64);      // qs is read before the next block reuses the tile
}

// Wide inputs (more 1024-blocks than rotating pairs in a CTA): one warp pair
// per block rotates x once for the whole grid and writes the operand words and
// group entries in the decode kernel's shared-memory layout.
__global__ void __launch_bounds__(64) ptq1_prep_kernel(const XSource xsrc, uint32_t groups, uint8_t *out) {
    __shared__ __align__(16) float tile[kRotScratch / 4];
    const int t = threadIdx.x;
    const uint32_t b = blockIdx.x;
    float d[16];
    if (xsrc.signs) load_signs16(xsrc, b, t, d);     // read-only parameter: before the dependency wait
    pdl_launch_dependents();
    pdl_wait();
    float v[16];
    load_run16(xsrc, b, t, v);
    int E;
    const int16_t *qs = rotate_quantize16(xsrc.signs != nullptr, t, v, d, tile, 1, &E);
    pack_ptq1(qs, out, groups, b, t, E, 1);
}

// sum_j t_j x16_j of one group: 24 base bytes (six words) and 2 high bytes,
// table lookups in lane-private copies, operand words from shared memory: the
// lane's copy of entry B sits at lut + (B << 7 | lane4), lane4 = 4 * lane.
__device__ __forceinline__ int group_dot(const uint32_t (&bw)[6], uint32_t hb, uint32_t lut, uint32_t lane4,
                                         const uint4 *aw) {
    uint4 a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = aw[i];
    const uint32_t *av = reinterpret_cast<const uint32_t *>(a);
    int acc[4] = {0, 0, 0, 0}, acc4 = 0;
#pragma unroll
    for (int q = 0; q < 6; ++q) {
        uint32_t W[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int sh = 8 * c - 7;
            const uint32_t off = ((sh >= 0 ? bw[q] >> sh : bw[q] << (-sh)) & 0x7F80u) | lane4;
            W[c] = lds32(lut + off);
            const uint32_t m = W[c] & 0x03030303u;
            const int j = 4 * q + c;
            acc[c] = dp2a_lo(av[2 * j], m, acc[c]);
            acc[c] = dp2a_hi(av[2 * j + 1], m, acc[c]);
        }
        // byte 0 of each entry holds 4 * t4 in bits 2-3: gather the four
        const uint32_t g = __byte_perm(__byte_perm(W[0], W[1], 0x0040u), __byte_perm(W[2], W[3], 0x0040u), 0x5410u) &
                           0x0C0C0C0Cu;
        acc4 = dp2a_lo(av[48 + 2 * q], g, acc4);
        acc4 = dp2a_hi(av[49 + 2 * q], g, acc4);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int sh = 8 * hh - 7;
        const uint32_t off = ((sh >= 0 ? hb >> sh : hb << (-sh)) & 0x7F80u) | lane4;
        const uint32_t m = lds32(lut + off) & 0x03030303u;
        acc[hh] = dp2a_lo(av[60 + 2 * hh], m, acc[hh]);
        acc[hh] = dp2a_hi(av[61 + 2 * hh], m, acc[hh]);
    }
    return acc[0] + acc[1] + acc[2] + acc[3] + (acc4 >> 2);
}

__global__ void __launch_bounds__(kThreads, 1) gemv_ptq1_int_kernel(const __grid_constant__ Ptq1Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const CtaRows cr = cta_rows(p);
    const bool last_cta = blockIdx.x == gridDim.x - 1;
    const uint32_t nitems = cr.nrb * p.nch;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t rem_bar = bar0 + 8 * kMaxSlots;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1;
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);      // the table starts the dynamic shared memory
    const uint32_t lut_s = smem_u32(smem), lane4 = 4u * (uint32_t)lane;
    uint8_t *rem_s = smem + p.off_rem;

    if (tid == 0) {
        prefetch_tmap(last_cta ? &p.bmap_last : &p.bmap_main);
        prefetch_tmap(last_cta ? &p.hmap_last : &p.hmap_main);
        prefetch_tmap(last_cta ? &p.smap_last : &p.smap_main);
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        mbar_init(rem_bar, 1);
        mbar_init(rem_bar + 8, 1);
        *failed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    const uint32_t pre = p.pre_issue < ring_to ? p.pre_issue : ring_to;
    if (tid == 0) {
        // weights are read-only parameters: a few items and the remainder rows before the dependency wait
        for (uint32_t i = 0; i < pre; ++i) issue_item(p, smem, i, last_cta);
        if (cr.rem) {
            const uint32_t rb_bytes = (uint32_t)(p.base_row + p.high_row + p.scale_row);
            mbar_arrive_expect_tx(rem_bar, cr.rem * rb_bytes);
            for (uint32_t rr = 0; rr < cr.rem; ++rr) {
                const uint64_t r = cr.begin + (uint64_t)cr.nrb * kRows + rr;
                const uint32_t d = smem_u32(rem_s) + rr * rb_bytes;
                bulk_g2s(d, p.base + r * p.base_row, (uint32_t)p.base_row, rem_bar);
                bulk_g2s(d + (uint32_t)p.base_row, p.high + r * p.high_row, (uint32_t)p.high_row, rem_bar);
                bulk_g2s(d + (uint32_t)(p.base_row + p.high_row), p.scale + r * p.scale_row, (uint32_t)p.scale_row,
                         rem_bar);
            }
        }
    }
    // digit table, replicated per bank: entry (B, l) at word 32 B + l; thread
    // tid computes entry tid / 2 and writes 16 of its copies
    {
        uint32_t B = (uint32_t)tid >> 1, W = 0;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint32_t t = B % 3;
            B /= 3;
            W |= i < 4 ? t << (8 * i) : t << 2;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(lut + (tid >> 1) * 32 + 16 * (tid & 1));
        const uint4 w4 = make_uint4(W, W, W, W);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = w4;
    }
    // rotation: warp pair pr = warp / 2 < nrot takes blocks pr, pr + nrot, ...
    // (none when the prep kernel has already written the operand words)
    const XSource xsrc{p.x, p.signs, p.k, p.x_dtype};
    const uint32_t nrot = p.act_g ? 0 : (p.nblk < kRotPairs ? p.nblk : kRotPairs);
    const uint32_t pr = warp >> 1;
    const int t = tid & 63;
    float d[16];
    if (p.signs && pr < nrot) load_signs16(xsrc, pr, t, d);     // also read-only
    pdl_launch_dependents();
    pdl_wait();          // x may come from the preceding kernel

    float v[16];
    if (pr < nrot) load_run16(xsrc, pr, t, v);
    uint8_t *act_s = smem + p.off_act;
    const uint32_t act_bar = rem_bar + 8;
    if (p.act_g && tid == 0) {          // the operand words, ahead of the rest of the ring
        mbar_arrive_expect_tx(act_bar, p.act_bytes);
        bulk_g2s(smem_u32(act_s), p.act_g, p.act_bytes, act_bar);
    }
    __syncthreads();     // every warp's x request is out: the rest of the ring queues behind them
    // the rest of the ring, one item per warp (lane 0 of warp w: items pre + w, pre + w + 16, ...)
    if (lane == 0)
        for (uint32_t i = pre + warp; i < ring_to; i += kWarps) issue_item(p, smem, i, last_cta);
    if (tid == 0) *issued = ring_to;
    if (pr < nrot) {
        float *tile = reinterpret_cast<float *>(smem + p.off_rot + pr * kRotScratch);
        for (uint32_t b = pr; b < p.nblk; b += nrot) {
            if (b != pr) {
                if (p.signs) load_signs16(xsrc, b, t, d);
                load_run16(xsrc, b, t, v);
            }
            int E;
            const int16_t *qs = rotate_quantize16(p.signs != nullptr, t, v, d, tile, 1 + pr, &E);
            pack_ptq1(qs, act_s, p.groups, b, t, E, 1 + pr);
        }
    }
    if (nrot) __syncthreads();      // the rotated operand words are complete (else they arrive on act_bar)

    bool ok = true;
    if (p.act_g) ok = mbar_wait(act_bar, 0, p.err);
    const uint32_t *act_w = reinterpret_cast<const uint32_t *>(act_s);
    const float2 *gs = reinterpret_cast<const float2 *>(act_s + (uint64_t)p.groups * kActStride * 4);
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    float *part_rem = part + kWarps * kRows;      // [kMaxRem][groups]

    // remainder rows: lanes = (row, group of the chunk); warp w takes chunks w, w + 16, ...
    if (cr.rem) {
        ok = ok && mbar_wait(rem_bar, 0, p.err);
        const uint32_t rb_bytes = (uint32_t)(p.base_row + p.high_row + p.scale_row);
        const uint32_t rr = lane >> 4;
        for (uint32_t ch = warp; ok && ch < p.nch; ch += kWarps) {
            const uint32_t G = ch * kChunk + (lane & 15);
            if (rr < cr.rem && G < p.groups) {
                const uint8_t *row = rem_s + rr * rb_bytes;
                const uint2 q0 = *reinterpret_cast<const uint2 *>(row + 24 * G);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(row + 24 * G + 8);
                const uint2 q2 = *reinterpret_cast<const uint2 *>(row + 24 * G + 16);
                const uint32_t bw[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
                const uint32_t hb = *reinterpret_cast<const uint16_t *>(row + p.base_row + 2 * G);
                const float s = __half2float(*reinterpret_cast<const __half *>(row + p.base_row + p.high_row + 2 * G));
                const float2 f = gs[G];
                const int dot = group_dot(bw, hb, lut_s, lane4, reinterpret_cast<const uint4 *>(act_w + G * kActStride));
                part_rem[rr * p.groups + G] = s * f.x * (float)(dot - __float_as_int(f.y));
            }
        }
    }

    // row blocks: warp w takes group 16 ch + w of item (rb, ch); lane = row
    const bool refill = nitems > p.nslots;
    uint32_t slot = 0, phase = 0, item = 0;
    // this warp's 24 bytes inside the item's 384-byte base run: three 8-byte words
    uint32_t boff[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const uint32_t o = 24 * warp + 8 * i, bx = o >> 7, c16 = (o & 127) >> 4, hf = (o >> 3) & 1;
        boff[i] = bx * kBaseBox + lane * 128 + ((c16 ^ (lane & 7)) << 4) + 8 * hf;
    }
    for (uint32_t rb = 0; rb < cr.nrb; ++rb) {
        float y = 0.f;
        for (uint32_t ch = 0; ch < p.nch; ++ch, ++item) {
            ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err);
            const uint32_t G = ch * kChunk + warp;
            if (ok && G < p.groups) {
                const uint8_t *sa = smem + p.off_ring + slot * kItemBytes;
                const uint2 q0 = *reinterpret_cast<const uint2 *>(sa + boff[0]);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(sa + boff[1]);
                const uint2 q2 = *reinterpret_cast<const uint2 *>(sa + boff[2]);
                const uint32_t bw[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
                const uint32_t hb = *reinterpret_cast<const uint16_t *>(sa + 3 * kBaseBox + lane * 32 + 2 * warp);
                const float s =
                    __half2float(*reinterpret_cast<const __half *>(sa + 3 * kBaseBox + 32 * kRows + lane * 32 + 2 * warp));
                const float2 f = gs[G];
                const int dot = group_dot(bw, hb, lut_s, lane4, reinterpret_cast<const uint4 *>(act_w + G * kActStride));
                y = fmaf(s * f.x, (float)(dot - __float_as_int(f.y)), y);
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
                            issue_item(p, smem, item + p.nslots, last_cta);
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
        part[warp * kRows + lane] = y;
        __syncthreads();
        if (warp == 0) {
            const uint32_t rl = rb * kRows + lane;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += part[w * kRows + lane];
            if (rl < cr.rows - cr.rem) store1(p.y, cr.begin + rl, p.y_dtype, acc);
        }
        __syncthreads();
    }
    if (cr.rem) {
        __syncthreads();       // part_rem complete (also when the CTA has no row-block pass)
        if (warp == 0 && lane < cr.rem) {
            float acc = 0.f;
            for (uint32_t G = 0; G < p.groups; ++G) acc += part_rem[lane * p.groups + G];
            store1(p.y, cr.begin + (uint64_t)cr.nrb * kRows + lane, p.y_dtype, acc);
        }
    }
    // after a timed-out wait: let the copies still in flight land (at most one
    // per slot, the last one issued into it) before the CTA's memory is freed
    if (tid == 0 && *(volatile uint32_t *)failed) {
        const uint32_t n_issued = *(volatile uint32_t *)issued;
        for (uint32_t i = n_issued > p.nslots ? n_issued - p.nslots : 0; i < n_issued; ++i)
            mbar_wait(bar0 + 8 * (i % p.nslots), (i / p.nslots) & 1, p.err, 200000000ll);
        if (cr.rem) mbar_wait(rem_bar, 0, p.err, 200000000ll);
        if (p.act_g) mbar_wait(rem_bar + 8, 0, p.err, 200000000ll);
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
    const uint32_t act_bytes = ((groups * (kActStride * 4 + 8) + 15) / 16) * 16;
    const bool split = nblk > kRotPairs;       // rotate in a separate kernel, once for the grid
    const uint32_t nrot = split ? 0 : std::min<uint32_t>(nblk, kRotPairs);
    const uint32_t rot_bytes = nrot * kRotScratch;
    const uint32_t rem_bytes = (uint32_t)(kMaxRem * (g.base_row_bytes + g.high_row_bytes + g.scale_row_bytes));
    const uint32_t part_bytes = (kWarps * kRows + kMaxRem * groups) * 4;
    const uint32_t bar_bytes = (kMaxSlots + 2) * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 4) * 4;
    const uint32_t fixed = kLutBytes + act_bytes + ((rot_bytes + 15) / 16) * 16 + ((rem_bytes + 15) / 16) * 16 +
                           ((part_bytes + 15) / 16) * 16 + bar_bytes + cnt_bytes;
    // with a prep kernel, leave room on the SM for one of its CTAs next to this kernel's
    const int limit = split ? smem_limit - 8 * 1024 : smem_limit;
    if ((int64_t)fixed + 2 * kItemBytes > limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((limit - (int)fixed) / (int)kItemBytes));
    // one CTA per SM with ~n / SMs rows each
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)sms, g.n / 32));
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid = (g.n + R - 1) / R;
    plan->ok = true;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nch = (groups + kChunk - 1) / kChunk;
    plan->nslots = nslots;
    plan->pre_issue = std::min<uint32_t>(1, nslots);
    uint32_t off = 0;
    plan->off_lut = off;         // fixed at 0: the kernel addresses the table from the start of its shared memory
    off += kLutBytes;
    plan->off_ring = off;
    off += nslots * kItemBytes;
    plan->off_act = off;
    off += act_bytes;
    plan->off_rot = off;
    off += ((rot_bytes + 15) / 16) * 16;
    plan->off_rem = off;
    off += ((rem_bytes + 15) / 16) * 16;
    plan->off_part = off;
    off += ((part_bytes + 15) / 16) * 16;
    plan->off_bar = off;
    off += bar_bytes;
    plan->off_cnt = off;
    off += cnt_bytes;
    plan->smem = off;
    plan->split = split;
    plan->act_bytes = act_bytes;
    plan->workspace = split ? act_bytes : 0;
    return true;
}

int gemv_ptq1_int_launch(const Ptq1Plan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, void *workspace,
                         cudaStream_t stream, bool pdl) {
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
    p.act_g = plan.split ? static_cast<const uint8_t *>(workspace) : nullptr;
    p.act_bytes = plan.act_bytes;
    p.y = y;
    p.n = g.n;
    p.k = (uint32_t)g.k;
    p.groups = (uint32_t)g.groups_per_row;
    p.nblk = (uint32_t)((g.k + 1023) / 1024);
    p.nch = plan.nch;
    p.rows_per_cta = plan.rows_per_cta;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.pre_issue = plan.pre_issue;
    p.off_ring = plan.off_ring;
    p.off_act = plan.off_act;
    p.off_rot = plan.off_rot;
    p.off_rem = plan.off_rem;
    p.off_part = plan.off_part;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_cta, G = plan.grid, last_rows = g.n - (G - 1) * R;
    if (G > 1) {
        st = encode_row_tiles(&p.bmap_main, p.base, g.base_row_bytes, R, G - 1, 128, kRows, true);
        if (!st) st = encode_row_tiles(&p.hmap_main, p.high, g.high_row_bytes, R, G - 1, 32, kRows, false);
        if (!st) st = encode_row_tiles(&p.smap_main, p.scale, g.scale_row_bytes, R, G - 1, 32, kRows, false);
        if (st) return st;
    }
    const uint64_t lr = (G - 1) * R;
    st = encode_rows(&p.bmap_last, p.base + lr * g.base_row_bytes, g.base_row_bytes, last_rows, 128, kRows, true);
    if (!st) st = encode_rows(&p.hmap_last, p.high + lr * g.high_row_bytes, g.high_row_bytes, last_rows, 32, kRows, false);
    if (!st)
        st = encode_rows(&p.smap_last, p.scale + lr * g.scale_row_bytes, g.scale_row_bytes, last_rows, 32, kRows, false);
    if (st) return st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    if (plan.split) {
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(p.nblk);
        pc.blockDim = dim3(64);
        pc.stream = stream;
        pc.attrs = attr;
        pc.numAttrs = 1;
        const XSource xsrc{x, signs, p.k, x_dtype};
        cudaError_t pe = cudaLaunchKernelEx(&pc, ptq1_prep_kernel, xsrc, p.groups, static_cast<uint8_t *>(workspace));
        if (pe != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 prep launch: %s", cudaGetErrorString(pe));
    }
    int st_attr = set_smem_attribute((const void *)gemv_ptq1_int_kernel, (int)plan.smem);
    if (st_attr) return st_attr;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_ptq1_int_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
