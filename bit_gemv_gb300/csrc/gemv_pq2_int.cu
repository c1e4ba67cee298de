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
// Activation: one warp per 1024-block rotates it in registers (the warp-held
// butterfly of device.cuh: five stages within the lane, five across lanes),
// takes the block maximum with shuffles and rounds to 16-bit fixed point,
// x16 = rint(v * 2^E) with max |x16| < 2^14, no shared-memory transpose and no
// barrier. A lane then holds 8 consecutive elements, which are exactly one
// 16-byte dp2a operand entry of the shared-memory activation table:
//   entry(word w, h) = {(x16[16w + 8h + p], x16[16w + 8h + 4 + p]), p = 0..3}.
//
// Arithmetic: in a 32-bit word of codes (16 weights, four per byte) the mask
// 0x03 << 2p per byte leaves the four codes of position p as bytes (times
// 4^p); dp2a multiplies two of them by two int16 activations and accumulates
// exactly in int32, one chain per position. Per group:
//   64 sum_j (code_j - 1) x16_j = ((acc0 * 4 + acc1) * 4 + acc2) * 4 + acc3
// where acc3 starts at -64 sum_j x16_j (exact in int32: |64 acc0| < 2^29),
// then y += scale * 2^-E / 64 * that, in fp32.
//
// Work: one CTA per SM owns a contiguous row range, in tiles of 128 rows.
// Weights stream through a ring of chunk slots; a chunk is 128 rows x 8
// groups: two 128-byte-swizzled tensor boxes of 128 rows x 128 bytes (a 3-D
// map view keeps them inside the CTA's rows) and one box of the rows' 8 scales
// (128 rows x 16 bytes), completing on the slot's mbarrier. The chunks of a
// tile are taken two at a time: warps 0-7 take chunk 2r and warps 8-15 chunk
// 2r + 1, warp w the whole group w % 8, lane l rows l, l+32, l+64, l+96, so
// each activation entry read from shared memory serves four rows. With an
// odd number of chunks per tile the last one is shared by all sixteen warps,
// half a group each. One chunk is requested before the programmatic-
// dependent-launch wait (weights and signs are read-only), the rest of the
// ring after x has arrived in the rotating warps (in a cluster, at once), by a
// warp that does not rotate; the last reader of a chunk refills its slot with the chunk nslots
// further on.
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "act16.cuh"
#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"
#include "rot2.cuh"

namespace ninfer {
namespace {

constexpr int kThreads = 512;     // 16 warps; one CTA per SM
constexpr int kWarps = 16;
constexpr int kRows = 128;        // rows per tile, four per lane
constexpr uint32_t kBoxBytes = 128 * kRows;               // one 128-byte column of the tile
constexpr uint32_t kChunkBytes = 2 * kBoxBytes + 16 * kRows;
constexpr uint32_t kMaxSlots = 8;
constexpr uint32_t kActGroupBytes = 256;                  // 16 operand entries per group
constexpr uint32_t kBarX = 1;                             // named barrier: x has arrived
constexpr uint32_t kBarPair0 = 2;                         // named barriers 2.. : one per rotating pair
constexpr uint32_t kMaxPairs = 7;                         // warps 0-13 (the producer, warp 15, never rotates)

struct IntParams {
    CUtensorMap wmap_main, wmap_last;   // base rows: {row bytes, R rows, CTA} / last CTA {row bytes, rows}
    CUtensorMap smap_main, smap_last;   // scale rows, same views
    CUtensorMap wmap2_main, wmap2_last, smap2_main, smap2_last;     // second matrix (fused gate/up: up)
    const void *x;
    const uint16_t *signs;              // bf16 +-1 per element, or null (no rotation)
    const uint16_t *signs2;             // second matrix's signs (may equal signs)
    uint32_t act_bytes;                 // operand entries + group entries of one rotation
    void *y;
    uint64_t n;
    uint32_t k, groups, nblk, nchunk, rows_per_cta;     // nchunk: chunks per tile and matrix, groups / 8
    int x_dtype, y_dtype;
    uint32_t nslots, pre_issue, nrot;    // nrot: warp pairs rotating at once (one scratch each)
    uint32_t nslots_inv;                 // floor(2^32 / nslots) + 1: item / nslots = umulhi(item, nslots_inv)
    uint32_t grid_rows;                  // CTAs with rows (the grid may have one more, for pairs)
    uint32_t off_ring, off_act, off_rot, off_part, off_bar, off_cnt;
    uint32_t *err;
    long long wait_cycles;              // bound of each ring wait
};

// Chunk i = tile * (kMats * nchunk) + mat * nchunk + j (groups 8j .. 8j + 7 of
// the tile's rows of matrix mat): its two weight boxes and its scale box into
// ring slot i % nslots (one thread).
template <int kMats>
__device__ __forceinline__ void issue_chunk(const IntParams &p, uint8_t *smem, uint32_t item, bool last_cta) {
    const uint32_t per_tile = kMats * p.nchunk;
    const uint32_t tile = item / per_tile, jj = item % per_tile, mat = kMats == 1 ? 0 : jj / p.nchunk;
    const uint32_t j = jj - mat * p.nchunk, slot = item % p.nslots;
    const uint32_t dst = smem_u32(smem + p.off_ring) + slot * kChunkBytes;
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    mbar_arrive_expect_tx(bar, kChunkBytes);
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

// Rotates block b with the pair (rotate_quant2) and writes its operand entries
// and group entries {2^-E / 64 (with the transform's 1/32), -64 * sum of x16}
// into act and, when act_remote is non-zero (the cluster address of the same
// table in the other CTA of the cluster), into that table too.
__device__ __forceinline__ void rotate_pack2(bool rotate, float (&v)[16], const float (&d)[16], uint32_t b,
                                             uint32_t groups, uint8_t *act, uint32_t act_remote, float *scr, int t,
                                             uint32_t bar) {
    const int lane = t & 31;
    uint32_t qb[16];
    const int E = rotate_quant2(rotate, v, d, scr, t, bar, qb);
    const float f = ldexpf(1.f, -E - 6 - (rotate ? 5 : 0));
    uint4 *ent = reinterpret_cast<uint4 *>(act);
    float2 *gs = reinterpret_cast<float2 *>(act + (uint64_t)groups * kActGroupBytes);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        // the run of elements 512 i + 8 t .. + 7: entry (t % 2) of word 32 i + t / 2 of the block,
        // group 4 i + t / 16 of the block; entry = {(x16[p], x16[4 + p]), p = 0..3}
        const uint32_t *q = qb + 8 * i;
        const uint32_t G = b * 8 + 4 * i + (t >> 4);
        uint4 en;
        en.x = __byte_perm(q[0], q[4], 0x5410);
        en.y = __byte_perm(q[1], q[5], 0x5410);
        en.z = __byte_perm(q[2], q[6], 0x5410);
        en.w = __byte_perm(q[3], q[7], 0x5410);
        if (G < groups) {
            ent[(uint64_t)b * 128 + 64 * i + t] = en;
            if (act_remote) st_cluster_v4(act_remote + (b * 128 + 64 * i + t) * 16, en);
        }
        // the group's sum of x16: the 16 lanes of each half-warp, one warp-wide add per half
        const int sum = (int)(q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7] - 8u * 0x4B400000u);
        const int s_lo = __reduce_add_sync(0xffffffffu, lane < 16 ? sum : 0);
        const int s_hi = __reduce_add_sync(0xffffffffu, lane < 16 ? 0 : sum);
        if ((lane & 15) == 0 && G < groups) {
            const int off = -64 * (lane < 16 ? s_lo : s_hi);
            gs[G] = make_float2(f, __int_as_float(off));
            if (act_remote) st_cluster_v2(act_remote + groups * kActGroupBytes + 8 * G, __float_as_uint(f), (uint32_t)off);
        }
    }
}

// kMats = 1: y = W x. kMats = 2 (fused FFN gate/up): y = silu(Wg x_g) * (Wu x_u)
// for the same rows of both matrices, x_g and x_u rotated with each matrix's
// signs. kXType: the dtype of x (one instance per dtype keeps the code short).
template <int kMats, int kXType>
__global__ void __launch_bounds__(kThreads, 1) gemv_pq2_int_kernel(const __grid_constant__ IntParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t r_begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t r_end = r_begin + p.rows_per_cta < p.n ? r_begin + p.rows_per_cta : p.n;
    const bool last_cta = blockIdx.x == p.grid_rows - 1;     // the last CTA with rows (an even grid may add one)
    const uint32_t per_tile = kMats * p.nchunk;
    const uint32_t ntile = r_end > r_begin ? (uint32_t)((r_end - r_begin + kRows - 1) / kRows) : 0;
    const uint32_t nitems = ntile * per_tile;
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + p.off_cnt);
    uint32_t *issued = cnt + kMaxSlots, *failed = cnt + kMaxSlots + 1;
    // rotation tasks (matrix, block): one rotation per block, or two when the
    // fused matrices have different signs. In a cluster of two CTAs each takes
    // every other task (local task i is task 2 i + rank) and writes the result
    // into both CTAs' tables.
    const uint32_t nrmat = (kMats == 2 && p.signs2 != p.signs) ? 2 : 1;
    const uint32_t ntask_all = nrmat * p.nblk;
    const uint32_t csize = cluster_nctarank(), crank = cluster_ctarank();
    const uint32_t ntask = csize == 2 ? (ntask_all + 1 - crank) / 2 : ntask_all;
    auto task_of = [&](uint32_t i) { return csize == 2 ? 2 * i + crank : i; };
    // the ring is issued by the last warp, which never rotates
    const int producer = kWarps - 1;
    const uint32_t ring_to = p.nslots < nitems ? p.nslots : nitems;
    const uint32_t pre = p.pre_issue < ring_to ? p.pre_issue : ring_to;
    // warp pairs rotate blocks: rotating pair pr takes tasks pr, pr + npr, ...
    const uint32_t npr = ntask < p.nrot ? ntask : p.nrot;       // rotating pairs, at most kMaxPairs
    const uint32_t pr = (uint32_t)warp >> 1;
    const int t = tid & 63;
    const bool rotating = pr < npr;
    const uint32_t nwait = 32 * (2 * npr + 1);
    // the rest of the ring is requested once x has arrived, except in a cluster
    // (two CTAs sharing the rotations), where requesting it at once measured faster
    const bool ring_after_x = csize == 1;

    if (tid == producer * 32) {
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
        // weights are read-only parameters: the first chunks before the dependency wait
        for (uint32_t i = 0; i < pre; ++i) issue_chunk<kMats>(p, smem, i, last_cta);
        *issued = pre;
    }
    uint8_t *act_s = smem + p.off_act;
    const uint32_t act_remote0 = csize == 2 ? mapa_shared(smem_u32(act_s), crank ^ 1u) : 0u;
    float v[16], d[16];
    if (rotating) {
        // the first rotation of a rotating pair
        const uint32_t task = task_of(pr);
        const uint32_t b = task % p.nblk;
        float *scr = reinterpret_cast<float *>(smem + p.off_rot + pr * kRotScratchBytes);
        if (p.signs) load_signs2(task >= p.nblk ? p.signs2 : p.signs, b, t, d);     // read-only
        pdl_launch_dependents();
        pdl_wait();          // x may come from the preceding kernel
        load_block2<kXType>(p.x, p.k, b, t, v);
        // x has arrived once its first and last values can be stored (in the
        // pair's maximum slot, written again later); then the producer may
        // queue the rest of the ring behind it
        *reinterpret_cast<volatile float *>(scr + 1080 + (t >> 5)) = v[0] + v[15];
        if (ring_after_x) named_barrier_arrive(kBarX, nwait);
        rotate_pack2(p.signs != nullptr, v, d, b, p.groups, act_s + (task / p.nblk) * p.act_bytes,
                     act_remote0 ? act_remote0 + (task / p.nblk) * p.act_bytes : 0u, scr, t, kBarPair0 + pr);
    } else {
        pdl_launch_dependents();
        pdl_wait();
        if (warp == producer) {
            // the rest of the ring is requested once x has arrived in every rotating
            // warp, so that x does not queue behind it
            if (ring_after_x) named_barrier(kBarX, nwait);
            if (lane == 0) {
                for (uint32_t i = pre; i < ring_to; ++i) issue_chunk<kMats>(p, smem, i, last_cta);
                *issued = ring_to;
            }
            __syncwarp();
        }
    }
    // more rotations than rotating pairs: further rounds
#pragma unroll 1
    for (uint32_t i = pr + npr; rotating && i < ntask; i += npr) {
        const uint32_t task = task_of(i), b = task % p.nblk;
        if (p.signs) load_signs2(task >= p.nblk ? p.signs2 : p.signs, b, t, d);
        load_block2<kXType>(p.x, p.k, b, t, v);
        rotate_pack2(p.signs != nullptr, v, d, b, p.groups, act_s + (task / p.nblk) * p.act_bytes,
                     act_remote0 ? act_remote0 + (task / p.nblk) * p.act_bytes : 0u,
                     reinterpret_cast<float *>(smem + p.off_rot + pr * kRotScratchBytes), t, kBarPair0 + pr);
    }
    // (the ring's barriers and counters, set up by the producer, are first used
    // after the barrier that completes the activation table)
    // the activation table is complete, in both CTAs of a cluster (this also
    // publishes the ring's barriers and counters to every warp)
    if (csize == 2) cluster_sync();
    else __syncthreads();

    bool ok = true;
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    const uint32_t gw = warp & 7, upper = warp >> 3;
    const uint32_t h = gw >> 2, gi = gw & 3;
    // swizzled 16-byte chunks (row % 8 pattern) of the group in column h's 128-byte line
    const uint32_t ch0 = ((2 * gi) ^ (lane & 7)) << 4, ch1 = ((2 * gi + 1) ^ (lane & 7)) << 4;
    const uint32_t rounds = (per_tile + 1) / 2;
#pragma unroll 1
    for (uint32_t tile = 0; tile < ntile; ++tile) {
        float y[kMats][4];      // rows lane + 32q of the tile, per matrix
#pragma unroll
        for (int mt = 0; mt < kMats; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q) y[mt][q] = 0.f;
#pragma unroll 1
        for (uint32_t r = 0; r < rounds; ++r) {
            // a full round: chunks 2r (warps 0-7) and 2r + 1 (warps 8-15), a whole group per warp;
            // the last round of an odd count: chunk 2r for all warps, half a group each
            const bool full = 2 * r + 1 < per_tile;
            const uint32_t jj = full ? 2 * r + upper : 2 * r;
            const uint32_t item = tile * per_tile + jj;
            const uint32_t cycle = __umulhi(item, p.nslots_inv);      // item / nslots (item < 2^29)
            const uint32_t slot = item - cycle * p.nslots, phase = cycle & 1;
            const uint32_t mat = kMats == 1 ? 0 : (jj >= p.nchunk), j = jj - mat * p.nchunk;
            const uint8_t *act_m = act_s + (mat < nrmat ? mat : 0) * p.act_bytes;
            const float2 *gs = reinterpret_cast<const float2 *>(act_m + (uint64_t)p.groups * kActGroupBytes);
            ok = ok && mbar_wait(bar0 + 8 * slot, phase, p.err, p.wait_cycles);
            const uint32_t G = j * 8 + gw;
            if (ok && G < p.groups) {
                const uint8_t *sa = smem + p.off_ring + slot * kChunkBytes;
                const uint8_t *wr = sa + h * kBoxBytes + lane * 128;
                const uint4 *aw = reinterpret_cast<const uint4 *>(act_m + (uint64_t)G * kActGroupBytes);
                const float2 f = gs[G];
                int acc[4][4];
                if (full) {
                    uint32_t w[4][8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(wr + q * 4096 + ch0);
                        const uint4 c = *reinterpret_cast<const uint4 *>(wr + q * 4096 + ch1);
                        w[q][0] = a.x; w[q][1] = a.y; w[q][2] = a.z; w[q][3] = a.w;
                        w[q][4] = c.x; w[q][5] = c.y; w[q][6] = c.z; w[q][7] = c.w;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[q][0] = 0; acc[q][1] = 0; acc[q][2] = 0; acc[q][3] = __float_as_int(f.y);
                    }
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
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
                } else {
                    // half a group: words 4 upper .. 4 upper + 3 (chunk 2 gi + upper of the line)
                    const uint32_t chh = upper ? ch1 : ch0;
                    uint32_t w[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(wr + q * 4096 + chh);
                        w[q][0] = a.x; w[q][1] = a.y; w[q][2] = a.z; w[q][3] = a.w;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[q][0] = 0; acc[q][1] = 0; acc[q][2] = 0; acc[q][3] = upper ? 0 : __float_as_int(f.y);
                    }
                    const uint4 *awh = aw + 8 * upper;
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint4 lo = awh[2 * wi], hi = awh[2 * wi + 1];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t c = w[q][wi];
                            acc[q][0] = dp2a_hi(hi.x, c & 0x03030303u, dp2a_lo(lo.x, c & 0x03030303u, acc[q][0]));
                            acc[q][1] = dp2a_hi(hi.y, c & 0x0C0C0C0Cu, dp2a_lo(lo.y, c & 0x0C0C0C0Cu, acc[q][1]));
                            acc[q][2] = dp2a_hi(hi.z, c & 0x30303030u, dp2a_lo(lo.z, c & 0x30303030u, acc[q][2]));
                            acc[q][3] = dp2a_hi(hi.w, c & 0xC0C0C0C0u, dp2a_lo(lo.w, c & 0xC0C0C0C0u, acc[q][3]));
                        }
                    }
                }
                // scale box: row r at r * 16 bytes holds the chunk's 8 scales
                const uint8_t *sc = sa + 2 * kBoxBytes + lane * 16 + 2 * gw;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t64 = ((acc[q][0] * 4 + acc[q][1]) * 4 + acc[q][2]) * 4 + acc[q][3];
                    const float s = __half2float(*reinterpret_cast<const __half *>(sc + q * 512));
                    if (kMats == 1 || mat == 0) y[0][q] = fmaf(s * f.x, (float)t64, y[0][q]);
                    else y[kMats - 1][q] = fmaf(s * f.x, (float)t64, y[kMats - 1][q]);
                }
            }
            // release the slot; its last reader (8 warps in a full round, 16 in the last
            // round of an odd count) refills it with the chunk nslots further on
            __syncwarp();
            if (lane == 0) {
                if (!ok) *failed = 1;
                __threadfence_block();
                const uint32_t seen = atomicAdd(&cnt[slot], 1u);
                if (seen == (full ? 7u : 15u)) {
                    cnt[slot] = 0;
                    if (ok && !*(volatile uint32_t *)failed && item + p.nslots < nitems) {
                        fence_proxy_async();
                        issue_chunk<kMats>(p, smem, item + p.nslots, last_cta);
                        atomicAdd(issued, 1u);
                    }
                }
            }
            __syncwarp();
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
    // chunk indices per CTA stay below 2^29 (the ring's slot arithmetic)
    if ((uint64_t)mats * (groups / 8) * ((g.n + 127) / 128) >= (1ull << 29)) return false;
    const uint32_t act_one = ((groups * (kActGroupBytes + 8) + 15) / 16) * 16;
    const uint32_t nrmat = (mats == 2 && two_rotations) ? 2 : 1;
    const uint32_t act_bytes = nrmat * act_one;
    const uint32_t part_bytes = mats * kWarps * kRows * 4;     // per-warp row sums of a tile (>= one scratch)
    const uint32_t bar_bytes = kMaxSlots * 8;
    const uint32_t cnt_bytes = (kMaxSlots + 4) * 4;
    // warp pairs rotating at once, each with its own scratch: as many as there
    // are rotations (at most kMaxPairs) while the ring keeps at least four slots
    // one CTA per SM with ~n / SMs rows each. When a CTA alone would need more
    // than one round of rotations, CTA pairs form clusters that share them (an
    // odd count gets one CTA without rows); otherwise the cluster's barrier
    // and paired scheduling would only add to the call.
    const uint64_t grid0 = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)sms, g.n / 64));
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid_rows = (g.n + R - 1) / R;
    const uint32_t ntask_all = nrmat * (uint32_t)((g.k + 1023) / 1024);
    const bool cluster = grid_rows >= 2 && ntask_all > kMaxPairs;
    const uint64_t grid = cluster ? (grid_rows + 1) / 2 * 2 : grid_rows;
    const uint32_t ntask = cluster ? (ntask_all + 1) / 2 : ntask_all;      // per CTA
    uint32_t nrot = std::min<uint32_t>(ntask, kMaxPairs);     // rotating warp pairs
    auto fixed_of = [&](uint32_t nr) { return act_bytes + nr * kRotScratchBytes + part_bytes + bar_bytes + cnt_bytes; };
    while (nrot > 1 && (int)fixed_of(nrot) + 4 * (int)kChunkBytes > smem_limit) nrot = (nrot + 1) / 2;
    const uint32_t fixed = fixed_of(nrot);
    if ((int)fixed + 2 * (int)kChunkBytes > smem_limit) return false;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (uint32_t)((smem_limit - (int)fixed) / (int)kChunkBytes));
    plan->ok = true;
    plan->grid_rows = (uint32_t)grid_rows;
    plan->cluster = cluster;
    plan->mats = mats;
    plan->act_one = act_one;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nitem = groups / 8;
    plan->nslots = nslots;
    plan->pre_issue = std::min<uint32_t>(1, nslots);
    plan->off_ring = 0;
    plan->off_act = nslots * kChunkBytes;
    plan->nrot = nrot;
    plan->off_rot = plan->off_act + act_bytes;
    plan->off_part = plan->off_rot + nrot * kRotScratchBytes;
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
    p.nchunk = plan.nitem;
    p.rows_per_cta = plan.rows_per_cta;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.nslots = plan.nslots;
    p.nslots_inv = (uint32_t)((1ull << 32) / plan.nslots + 1);
    p.grid_rows = plan.grid_rows;
    p.pre_issue = plan.pre_issue;
    p.off_ring = plan.off_ring;
    p.off_act = plan.off_act;
    p.nrot = plan.nrot;
    p.off_rot = plan.off_rot;
    p.off_part = plan.off_part;
    p.off_bar = plan.off_bar;
    p.off_cnt = plan.off_cnt;
    p.wait_cycles = wait_limit_cycles();
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_cta, G = plan.grid_rows, last_rows = g.n - (G - 1) * R;
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
    void (*kernel)(IntParams) = nullptr;
    if (x_dtype == NINFER_F32) kernel = plan.mats == 2 ? gemv_pq2_int_kernel<2, NINFER_F32> : gemv_pq2_int_kernel<1, NINFER_F32>;
    else if (x_dtype == NINFER_BF16)
        kernel = plan.mats == 2 ? gemv_pq2_int_kernel<2, NINFER_BF16> : gemv_pq2_int_kernel<1, NINFER_BF16>;
    else kernel = plan.mats == 2 ? gemv_pq2_int_kernel<2, NINFER_F16> : gemv_pq2_int_kernel<1, NINFER_F16>;
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
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer
