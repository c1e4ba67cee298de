// Decode GEMV for PTQ1_0_G128 weights and 1 <= M <= 8 activation rows on the
// binary16 mma.sync tensor path, split over the 1024-blocks of k.
//
// What it computes:
//   y[m][r] = sum_g scale[r][g] * sum_{j<128} (t[r][128g+j] - 1) * xr[m][128g+j]
// with xr the forward-rotated activation (per 1024-block H (D * x) / 32,
// "artifact-container.md" §8 hadamard_signs; TensorSharp article §4.2) and t
// the base-3 digits of the planes ("bonsai三元GGUF模型转ninfer模型01" §3-§4): base
// byte j of a group holds weights 5j .. 5j+4 as (byte / 3^i) % 3, high byte h
// holds weights 120 + 4h .. 123 + 4h; one binary16 scale per group.
//
// Work split: CTA (b, t) takes 1024-block b of k (groups 8b .. 8b + 7) for the
// rows of row tile t. Every CTA therefore rotates a single block of x (one warp
// pair per activation row), and blocks x tiles fill the SMs even when n is
// small. With more than one block each CTA stores its fp32 partial sums
// P[b][m][r]; ptq1_reduce_kernel adds the blocks in order and stores y.
//
// Arithmetic: mma.sync m16n8k16, binary16 operands, fp32 accumulate; the eight
// MMA columns are the activation rows.
//  * A (digits): a 256-entry table maps a code byte to
//      t0 | t4 << 2 | t2 << 8 | t1 << 16 | t3 << 24,
//    kept in 32 lane-private copies (lane l always reads bank l). Masking gives
//    (t0, t1) and a byte permute (t2, t3) as binary16 subnormals t * 2^-24;
//    t4 of two bytes is pulled from bits 2-3 of their entries.
//  * K order inside a group (any permutation works as long as A and B agree):
//    lane c of a quad owns base bytes c, c + 4, ..., c + 20 (byte c of each
//    base word). k-steps 0-5 hold digits 0-3 of byte 4s + c at the lane's four
//    K slots; step 6 holds t4 of bytes c, c + 4, c + 8, c + 12; step 7 holds t4
//    of bytes c + 16, c + 20 and digits 2 (c % 2), 2 (c % 2) + 1 of high byte c / 2.
//  * B: binary16 xr * 2^E (E per block and activation row, max |.| < 2^11)
//    in that K order, written once per CTA into shared memory and kept in
//    registers by the warps.
//  * Per group: acc += scale * (2^24 * C - X), X = sum of the group's B
//    (value = t - 1); acc * 2^-E when the item is stored.
// Products of binary16 operands are exact; the sums are fp32.
//
// Data movement: items of 128 rows x 8 groups (two 96-byte boxes of base bytes,
// one 16-byte box of high bytes and one of scales) stream through a ring of TMA
// slots on mbarriers; all of a CTA's items are requested before the dependency
// wait when they fit. Warp w takes the 16-row slice w / 2 and the four groups
// 4 (w % 2) .. 4 (w % 2) + 3; the two warps of a slice add their halves through
// shared memory.
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
constexpr int kRows = 128;        // rows per item: 8 slices of 16
constexpr uint32_t kBaseBox = 96 * kRows;                  // base bytes of 4 groups
constexpr uint32_t kSideBox = 16 * kRows;                  // high bytes (or scales) of 8 groups
constexpr uint32_t kItemBytes = 2 * kBaseBox + 2 * kSideBox;
constexpr uint32_t kMaxSlots = 6;
constexpr uint32_t kPairs = 8;                             // rotating warp pairs: one per activation row
constexpr uint32_t kLutBytes = 256 * 32 * 4;
constexpr uint32_t kFragBytes = 8 * 8 * 32 * 8;            // 8 groups x 8 k-steps x 32 lanes x 2 registers
constexpr uint32_t kFxBytes = (8 * 8 + 8) * 4;             // X per (group, row), then 2^-E per row
constexpr uint32_t kPartBytes = 2 * 8 * 32 * 16;           // double-buffered float4 per lane of the odd warps
constexpr uint32_t kRotBytes = kPairs * kRotScratch;         // rotation tiles; then the slice partials
static_assert(kPartBytes <= kRotBytes, "slice partials live in the rotation tiles");
constexpr bool kHoldB = true;     // keep the warp's B fragments in registers (else read them per k-step)
constexpr bool kSplitC = false;   // two accumulator chains per group (even / odd k-steps)

struct Ptq1MmaParams {
    CUtensorMap bmap_main, bmap_last;   // base rows {row bytes, R rows, tile} / last tile {row bytes, rows}
    CUtensorMap hmap_main, hmap_last;   // high rows, same views
    CUtensorMap smap_main, smap_last;   // scale rows, same views
    const void *x;
    const uint16_t *signs;
    float *part;                        // P[b][m][r], r stride n_pad; null with one block (y stored directly)
    void *y;
    uint64_t n, n_pad, x_row_bytes;
    uint32_t k, M, rows_per_tile;
    int x_dtype, y_dtype;
    uint32_t nslots;
    uint32_t off_ring, off_lut, off_rot, off_frag, off_bar, off_cnt;
    uint32_t *err;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// Digit-table entry of code byte B.
__device__ __forceinline__ uint32_t digit_entry(uint32_t B) {
    uint32_t t[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        t[i] = B % 3;
        B /= 3;
    }
    return t[0] | t[4] << 2 | t[2] << 8 | t[1] << 16 | t[3] << 24;
}

__device__ __forceinline__ uint32_t digits01(uint32_t e) { return e & 0x00030003u; }               // (t0, t1)
__device__ __forceinline__ uint32_t digits23(uint32_t e) { return __byte_perm(e, 0u, 0x4341); }    // (t2, t3)
__device__ __forceinline__ uint32_t digits44(uint32_t ea, uint32_t eb) {                           // (t4 of a, t4 of b)
    return (__byte_perm(ea, eb, 0x5410) >> 2) & 0x00030003u;
}

// Item i of the CTA's tile (rows 128 i .. 128 i + 127 of the tile, groups of
// block b) into ring slot i % nslots (one thread).
__device__ __forceinline__ void issue_item(const Ptq1MmaParams &p, uint8_t *smem, uint32_t item, uint32_t b,
                                           bool last_tile) {
    const uint32_t slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kItemBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kItemBytes);
    const int y0 = (int)(item * kRows), z = (int)blockIdx.y;
    const int xb = (int)(192 * b), xs = (int)(16 * b);
    if (last_tile) {
        tma_load_2d(dst, &p.bmap_last, xb, y0, bar);
        tma_load_2d(dst + kBaseBox, &p.bmap_last, xb + 96, y0, bar);
        tma_load_2d(dst + 2 * kBaseBox, &p.hmap_last, xs, y0, bar);
        tma_load_2d(dst + 2 * kBaseBox + kSideBox, &p.smap_last, xs, y0, bar);
    } else {
        tma_load_3d(dst, &p.bmap_main, xb, y0, z, bar);
        tma_load_3d(dst + kBaseBox, &p.bmap_main, xb + 96, y0, z, bar);
        tma_load_3d(dst + 2 * kBaseBox, &p.hmap_main, xs, y0, z, bar);
        tma_load_3d(dst + 2 * kBaseBox + kSideBox, &p.smap_main, xs, y0, z, bar);
    }
}

__global__ void __launch_bounds__(kThreads, 1) gemv_ptq1_mma_kernel(const __grid_constant__ Ptq1MmaParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b = blockIdx.x;
    const bool last_tile = blockIdx.y == gridDim.y - 1;
    const uint64_t r_begin = (uint64_t)blockIdx.y * p.rows_per_tile;
    const uint64_t r_end = r_begin + p.rows_per_tile < p.n ? r_begin + p.rows_per_tile : p.n;
    const uint32_t rows = (uint32_t)(r_end - r_begin);
    const uint32_t nitems = (rows + kRows - 1) / kRows;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1;

    if (tid == 0) {
        prefetch_tmap(last_tile ? &p.bmap_last : &p.bmap_main);
        prefetch_tmap(last_tile ? &p.hmap_last : &p.hmap_main);
        prefetch_tmap(last_tile ? &p.smap_last : &p.smap_main);
        for (uint32_t s = 0; s < p.nslots; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            cnt[s] = 0;
        }
        *failed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    if (tid == 0) {
        // weights are read-only parameters: the whole ring before the dependency wait
        for (uint32_t i = 0; i < ring_to; ++i) issue_item(p, smem, i, b, last_tile);
        *issued = ring_to;
    }

    // digit table, lane-private copies: entry (B, l) at word 32 B + l; thread
    // tid computes entry tid / 2 and writes 16 of its copies (before the
    // dependency wait: it depends on nothing)
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem + p.off_lut);
    {
        const uint32_t W = digit_entry((uint32_t)tid >> 1);
        uint4 *dst = reinterpret_cast<uint4 *>(lut + (tid >> 1) * 32 + 16 * (tid & 1));
        const uint4 w4 = make_uint4(W, W, W, W);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = w4;
    }
    // B fragments of block b: warp pair m rotates activation row m into
    // binary16 (natural order, in its own rotation tile), then all threads
    // gather the fragments from those rows
    const uint32_t m = warp >> 1;
    const int t = tid & 63;
    const XSource xsrc{p.x, p.signs, p.k, p.x_dtype};
    float d[16];
    if (p.signs && m < p.M) load_signs16(xsrc, b, t, d);     // read-only parameter: before the dependency wait
    pdl_launch_dependents();
    pdl_wait();          // x may come from the preceding kernel
    float *fx = reinterpret_cast<float *>(smem + p.off_frag + kFragBytes);     // X[g * 8 + m], then 2^-E[m]
    {
        float *tile = reinterpret_cast<float *>(smem + p.off_rot + m * kRotScratch);
        float v[16];
        int E = 0;
        if (m < p.M) {
            XSource xs = xsrc;
            xs.x = static_cast<const uint8_t *>(p.x) + m * p.x_row_bytes;
            load_run16(xs, b, t, v);
            const float mx = rotate16(p.signs != nullptr, t, v, d, tile, 1 + m);
            if (mx > 0.f) E = 10 - ilogbf(mx);      // max |xr * 2^E| < 2^11
            E = max(-100, min(100, E));
        } else {
#pragma unroll
            for (int r = 0; r < 16; ++r) v[r] = 0.f;
        }
        // v[r] is element 256 (r / 4) + 4t + r % 4 of the block (group 2 (r / 4) + t / 32)
        const float up = ldexpf(1.f, E);
        uint2 *row = reinterpret_cast<uint2 *>(tile);     // 1024 binary16, elements 4j .. 4j + 3 per uint2
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            __half h[4];
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[i] = __float2half_rn(v[4 * a + i] * up);
                sum += __half2float(h[i]);
            }
            row[64 * a + t] = make_uint2((uint32_t)__half_as_ushort(h[0]) | (uint32_t)__half_as_ushort(h[1]) << 16,
                                         (uint32_t)__half_as_ushort(h[2]) | (uint32_t)__half_as_ushort(h[3]) << 16);
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
            if (lane == 0) fx[(2 * a + (t >> 5)) * 8 + m] = sum;
        }
        if (t == 0) fx[64 + m] = m < p.M ? ldexpf(1.f, -E) : 0.f;
    }
    __syncthreads();     // binary16 rows complete
    {
        // fragment word u = (g * 8 + s) * 32 + lane of column m = lane / 4, quad lane c
        // = lane % 4: the weights that the group's K order (above) puts at k-step s,
        // slots 2c, 2c + 1, 2c + 8, 2c + 9
        uint2 *fw = reinterpret_cast<uint2 *>(smem + p.off_frag);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = (uint32_t)tid + 512 * i, s = (u >> 5) & 7, g = u >> 8, mm = lane >> 2, c = lane & 3;
            const uint16_t *st = reinterpret_cast<const uint16_t *>(smem + p.off_rot + mm * kRotScratch) + 128 * g;
            uint32_t w[4];
            if (s < 6) {
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = st[20 * s + 5 * c + q];
            } else if (s == 6) {
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = st[5 * c + 20 * q + 4];
            } else {
                w[0] = st[5 * c + 84];
                w[1] = st[5 * c + 104];
                w[2] = st[120 + 2 * c];
                w[3] = st[121 + 2 * c];
            }
            fw[u] = make_uint2(w[0] | w[1] << 16, w[2] | w[3] << 16);
        }
    }
    __syncthreads();     // fragments complete; the rotation tiles are free (they hold the slice partials next)
    uint16_t *frag = reinterpret_cast<uint16_t *>(smem + p.off_frag);
    const uint32_t slice = warp >> 1, gh = warp & 1, g4 = lane >> 2, c = lane & 3;
    // this warp's B fragments (groups 4 gh .. 4 gh + 3), X and 2^-E of columns 2c, 2c + 1
    uint2 bfr[4][8];
    float X0[4], X1[4];
    const uint2 *fw = reinterpret_cast<const uint2 *>(frag) + (4 * gh) * 8 * 32 + lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (kHoldB) {
#pragma unroll
            for (int s = 0; s < 8; ++s) bfr[q][s] = fw[(q * 8 + s) * 32];
        }
        X0[q] = fx[(4 * gh + q) * 8 + 2 * c];
        X1[q] = fx[(4 * gh + q) * 8 + 2 * c + 1];
    }
    const float sc0 = fx[64 + 2 * c], sc1 = fx[64 + 2 * c + 1];

    const uint32_t *lutl = lut + lane;        // lane-private copy: entry B at lutl[32 B]
    const uint32_t selc = 0x4440u | c;          // byte c of a word to byte 0, zeros above
    const uint32_t selh = (c & 1) ? 0x4341u : 0x4240u;     // digits (t2, t3) or (t0, t1) of a high byte
    float4 *part = reinterpret_cast<float4 *>(smem + p.off_rot);
    const bool refill = nitems > p.nslots;
    bool ok = true;
    uint32_t slot = 0, phase = 0;
    for (uint32_t it = 0; it < nitems; ++it) {
        ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};      // rows g4, g4 + 8 of the slice x columns 2c, 2c + 1
        const uint32_t item_rows = rows - it * kRows;
        if (ok && slice * 16 < item_rows) {
            const uint8_t *sb = smem + p.off_ring + slot * kItemBytes;
            const uint32_t rA = slice * 16 + g4;
            const uint8_t *baseA = sb + gh * kBaseBox + rA * 96, *baseB = baseA + 8 * 96;
            const uint8_t *sideA = sb + 2 * kBaseBox + rA * 16, *sideB = sideA + 8 * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t gl = 4 * gh + q;
                // the group's 24 base bytes of rows A and B: one 16-byte and one 8-byte load each
                uint32_t wA[6], wB[6];
                {
                    const int o16 = (q & 1) ? 8 : 0, o8 = (q & 1) ? 0 : 16;     // 24q is 16-aligned for even q
                    const uint4 a4 = *reinterpret_cast<const uint4 *>(baseA + 24 * q + o16);
                    const uint4 b4 = *reinterpret_cast<const uint4 *>(baseB + 24 * q + o16);
                    const uint2 a2 = *reinterpret_cast<const uint2 *>(baseA + 24 * q + o8);
                    const uint2 b2 = *reinterpret_cast<const uint2 *>(baseB + 24 * q + o8);
                    const int w16 = o16 / 4, w8 = o8 / 4;
                    wA[w16] = a4.x; wA[w16 + 1] = a4.y; wA[w16 + 2] = a4.z; wA[w16 + 3] = a4.w;
                    wB[w16] = b4.x; wB[w16 + 1] = b4.y; wB[w16 + 2] = b4.z; wB[w16 + 3] = b4.w;
                    wA[w8] = a2.x; wA[w8 + 1] = a2.y;
                    wB[w8] = b2.x; wB[w8 + 1] = b2.y;
                }
                uint32_t eA[6], eB[6];
                float C[4] = {0.f, 0.f, 0.f, 0.f}, D[4] = {0.f, 0.f, 0.f, 0.f};
                auto bf = [&](int st) { return kHoldB ? bfr[q][st] : fw[(q * 8 + st) * 32]; };
#pragma unroll
                for (int st = 0; st < 6; ++st) {
                    eA[st] = lutl[__byte_perm(wA[st], 0u, selc) << 5];
                    eB[st] = lutl[__byte_perm(wB[st], 0u, selc) << 5];
                    mma16816(kSplitC && (st & 1) ? D : C, digits01(eA[st]), digits01(eB[st]), digits23(eA[st]),
                             digits23(eB[st]), bf(st));
                }
                mma16816(C, digits44(eA[0], eA[1]), digits44(eB[0], eB[1]), digits44(eA[2], eA[3]),
                         digits44(eB[2], eB[3]), bf(6));
                const uint32_t hA = lutl[(uint32_t)sideA[2 * gl + (c >> 1)] << 5];
                const uint32_t hB = lutl[(uint32_t)sideB[2 * gl + (c >> 1)] << 5];
                mma16816(kSplitC ? D : C, digits44(eA[4], eA[5]), digits44(eB[4], eB[5]),
                         __byte_perm(hA, 0u, selh) & 0x00030003u, __byte_perm(hB, 0u, selh) & 0x00030003u, bf(7));
                if (kSplitC) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) C[i] += D[i];
                }
                const float sA = __half2float(*reinterpret_cast<const __half *>(sideA + kSideBox + 2 * gl));
                const float sB = __half2float(*reinterpret_cast<const __half *>(sideB + kSideBox + 2 * gl));
                acc[0] = fmaf(sA, fmaf(C[0], 16777216.f, -X0[q]), acc[0]);
                acc[1] = fmaf(sA, fmaf(C[1], 16777216.f, -X1[q]), acc[1]);
                acc[2] = fmaf(sB, fmaf(C[2], 16777216.f, -X0[q]), acc[2]);
                acc[3] = fmaf(sB, fmaf(C[3], 16777216.f, -X1[q]), acc[3]);
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
                        issue_item(p, smem, it + p.nslots, b, last_tile);
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
        // the two warps of a slice hold complementary group halves: add them and store
        float4 *pb = part + ((it & 1) * 8 + slice) * 32 + lane;
        if (gh) *pb = make_float4(acc[0], acc[1], acc[2], acc[3]);
        named_barrier(1 + slice, 64);
        if (!gh) {
            const float4 o = *pb;
            const float sum[4] = {(acc[0] + o.x) * sc0, (acc[1] + o.y) * sc1, (acc[2] + o.z) * sc0,
                                  (acc[3] + o.w) * sc1};
            const uint32_t rl = it * kRows + slice * 16 + g4;     // tile-local rows rl, rl + 8
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t r = rl + 8 * (i >> 1), mm = 2 * c + (i & 1);
                if (r < rows && mm < p.M) {
                    const uint64_t row = r_begin + r;
                    if (p.part) p.part[((uint64_t)b * p.M + mm) * p.n_pad + row] = sum[i];
                    else store1(p.y, (uint64_t)mm * p.n + row, p.y_dtype, sum[i]);
                }
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
    }
}

// y[m][r] = sum over blocks b (in order) of P[b][m][r]; two rows per thread,
// with up to 32 blocks' loads in flight before their sums.
__global__ void __launch_bounds__(128) ptq1_reduce_kernel(const float *part, uint32_t nblk, uint32_t M, uint64_t n,
                                                          uint64_t n_pad, void *y, int y_dtype) {
    pdl_launch_dependents();
    pdl_wait();          // the partial sums come from the preceding kernel
    const uint64_t per_m = n_pad / 2;
    const uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= (uint64_t)M * per_m) return;
    const uint32_t m = (uint32_t)(q / per_m);
    const uint64_t j = q % per_m;
    const float2 *src = reinterpret_cast<const float2 *>(part) + (uint64_t)m * per_m + j;
    const uint64_t bstride = (uint64_t)M * per_m;
    float2 s = make_float2(0.f, 0.f);
    for (uint32_t bb = 0; bb < nblk; bb += 32) {
        float2 v[32];
#pragma unroll
        for (uint32_t i = 0; i < 32; ++i)
            if (bb + i < nblk) v[i] = __ldcg(src + (uint64_t)(bb + i) * bstride);
#pragma unroll
        for (uint32_t i = 0; i < 32; ++i) {
            if (bb + i < nblk) {
                s.x += v[i].x;
                s.y += v[i].y;
            }
        }
    }
    if (2 * j < n) store1(y, (uint64_t)m * n + 2 * j, y_dtype, s.x);
    if (2 * j + 1 < n) store1(y, (uint64_t)m * n + 2 * j + 1, y_dtype, s.y);
}

}  // namespace

bool gemv_ptq1_mma_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                        Ptq1MmaPlan *plan) {
    *plan = Ptq1MmaPlan{};
    if (M < 1 || M > kPairs) return false;
    if (rotate && g.k % 1024) return false;
    if (g.k % 8) return false;     // rows of x after the first stay 16-byte aligned for the vector loads
    // boxes are whole 1024-blocks: base rows 192 bytes, high and scale rows 16 bytes per block
    if (g.groups_per_row % 8 || g.base_row_bytes != 24 * g.groups_per_row || g.high_row_bytes != 2 * g.groups_per_row ||
        g.scale_row_bytes != 2 * g.groups_per_row)
        return false;
    if (g.k > (1u << 24) || g.n > (1ull << 31) || g.n == 0) return false;
    const uint32_t nblk = (uint32_t)(g.groups_per_row / 8);
    // tiles: about SMs / blocks of them, each a multiple of 16 rows
    uint64_t T = std::max<uint64_t>(1, (uint64_t)sms / nblk);
    T = std::min<uint64_t>(T, (g.n + 15) / 16);
    const uint64_t R = ((g.n + T - 1) / T + 15) / 16 * 16;
    T = (g.n + R - 1) / R;
    const uint32_t nitem = (uint32_t)((R + kRows - 1) / kRows);
    const uint32_t bar_bytes = kMaxSlots * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 4) * 4;
    const uint32_t fixed = kLutBytes + kRotBytes + kFragBytes + kFxBytes + bar_bytes + cnt_bytes;
    if ((int64_t)fixed + kItemBytes > smem_limit) return false;
    uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((smem_limit - (int)fixed) / (int)kItemBytes));
    nslots = std::min(nslots, nitem);
    if (nslots < 2 && nitem > 1) return false;
    plan->ok = true;
    plan->nblk = nblk;
    plan->tiles = (uint32_t)T;
    plan->rows_per_tile = (uint32_t)R;
    plan->nslots = nslots;
    uint32_t off = 0;
    plan->off_ring = off;
    off += nslots * kItemBytes;
    plan->off_lut = off;
    off += kLutBytes;
    plan->off_rot = off;
    off += kRotBytes;
    plan->off_frag = off;
    off += kFragBytes + kFxBytes;
    plan->off_bar = off;
    off += bar_bytes;
    plan->off_cnt = off;
    off += cnt_bytes;
    plan->smem = off;
    plan->n_pad = (g.n + 3) / 4 * 4;
    plan->workspace = nblk > 1 ? (uint64_t)nblk * M * plan->n_pad * sizeof(float) : 0;
    return true;
}

int gemv_ptq1_mma_launch(const Ptq1MmaPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g,
                         const void *x, int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M,
                         void *workspace, cudaStream_t stream, bool pdl) {
    Ptq1MmaParams p;
    std::memset(&p, 0, sizeof p);
    const uint8_t *base = payload + g.base_offset, *high = payload + g.high_offset, *scale = payload + g.scale_offset;
    p.x = x;
    p.signs = signs;
    p.part = plan.nblk > 1 ? static_cast<float *>(workspace) : nullptr;
    p.y = y;
    p.n = g.n;
    p.n_pad = plan.n_pad;
    p.x_row_bytes = g.k * dtype_size(x_dtype);
    p.k = (uint32_t)g.k;
    p.M = (uint32_t)M;
    p.rows_per_tile = plan.rows_per_tile;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.off_ring = plan.off_ring;
    p.off_lut = plan.off_lut;
    p.off_rot = plan.off_rot;
    p.off_frag = plan.off_frag;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_tile, T = plan.tiles, lr = (T - 1) * R, last_rows = g.n - lr;
    if (T > 1) {
        st = encode_row_tiles(&p.bmap_main, base, g.base_row_bytes, R, T - 1, 96, kRows, false);
        if (!st) st = encode_row_tiles(&p.hmap_main, high, g.high_row_bytes, R, T - 1, 16, kRows, false);
        if (!st) st = encode_row_tiles(&p.smap_main, scale, g.scale_row_bytes, R, T - 1, 16, kRows, false);
        if (st) return st;
    }
    st = encode_rows(&p.bmap_last, base + lr * g.base_row_bytes, g.base_row_bytes, last_rows, 96, kRows, false);
    if (!st) st = encode_rows(&p.hmap_last, high + lr * g.high_row_bytes, g.high_row_bytes, last_rows, 16, kRows, false);
    if (!st)
        st = encode_rows(&p.smap_last, scale + lr * g.scale_row_bytes, g.scale_row_bytes, last_rows, 16, kRows,
                         false);
    if (st) return st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    int st_attr = set_smem_attribute((const void *)gemv_ptq1_mma_kernel, (int)plan.smem);
    if (st_attr) return st_attr;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.nblk, plan.tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_ptq1_mma_kernel, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 mma gemv launch: %s", cudaGetErrorString(e));
    if (plan.nblk > 1) {
        const uint64_t threads = M * plan.n_pad / 2;
        cudaLaunchConfig_t rc = {};
        rc.gridDim = dim3((unsigned)((threads + 127) / 128));
        rc.blockDim = dim3(128);
        rc.stream = stream;
        rc.attrs = attr;
        rc.numAttrs = 1;
        e = cudaLaunchKernelEx(&rc, ptq1_reduce_kernel, static_cast<const float *>(workspace), plan.nblk, (uint32_t)M,
                               (uint64_t)g.n, plan.n_pad, y, y_dtype);
        if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "ptq1 block reduction launch: %s", cudaGetErrorString(e));
    }
    return NINFER_OK;
}

}  // namespace ninfer
