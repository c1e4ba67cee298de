// Fused rotate + decode + GEMV for PQ2_0_G128 weights, 2 <= M <= 8 activation rows.
//
// What it computes (the decode projection):
//   y[m][r] = sum_g scale[r][g] * sum_{j<128} (code[r][128g+j] - 1) * xr[m][128g+j],
//   xr = per-1024-block H (D * x) / 32 ("artifact-container.md" §8 hadamard_signs;
//   TensorSharp article §4.2), codes = 2-bit fields of the base plane, least
//   significant first, value = code - 1 ("GGUF 完整讲解" §4.3), one binary16 scale
//   per 128-weight group at scale_offset ("bonsai三元GGUF模型转ninfer模型01" §3).
//
// How (GB300 design):
//  * One CTA per SM owns a contiguous row range. Its weight rows stream from HBM
//    into shared-memory slots (32 rows each) with one bulk async copy per row
//    (rows padded so the MMA operand reads are bank-conflict free) plus one copy
//    of the tile's scales, all completing on an mbarrier. The copies are issued
//    before the programmatic-dependent-launch wait: weights never depend on the
//    preceding kernel, so the next projection's weight stream overlaps the
//    previous one's tail.
//  * Every CTA rotates the activation itself (a 1024-point butterfly per block
//    held by one warp) and writes it to shared memory as a three-term e4m3
//    expansion xr*2^E ~ t0 + t1/16 + t2/256 (E per block and token), already in
//    the m16n8k32 B-fragment order. Column 3m+q of the MMA holds term q of token m.
//  * Decode: a code c sits in bits 2p..2p+1 of a byte; masking a 32-bit word
//    with 0x03030303 / 0x0C0C0C0C (after an optional >>4) leaves four e4m3
//    subnormals c*2^-9 (or 4c*2^-9) - exact - so one LOP3 yields four A
//    operands. The factor 4 of odd positions is divided out of the B terms.
//  * The e4m3 tensor core sums sum_j c_j * t_q(xr_j) exactly into fp32; per
//    group, y += scale * (F * P - O) with F = 2^(9-E-4q) and O the group's
//    sum of B terms (the "-1" of the offset code), still fp32.
// One activation row runs on the integer pipes instead (gemv_pq2_int.cu); with
// several rows one decoded A fragment serves all of them, which the integer
// path cannot share.
#include <cstring>

#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "async.cuh"
#include "common.h"
#include "device.cuh"
#include "gemv.h"

namespace ninfer {

namespace {

constexpr int kTile = 32;        // rows per slot / warp-pair tile
constexpr int kMaxSlots = 4;

struct Params {
    CUtensorMap tmap_main;  // base plane as {row bytes, R rows, CTA} (CTAs 0 .. G-2)
    CUtensorMap tmap_last;  // base rows of the last CTA as {row bytes, rows}
    const uint8_t *base;    // base plane
    const uint8_t *scale;   // scale plane
    const void *x;
    const uint16_t *signs;  // nullptr: no rotation
    void *y;
    uint64_t n;
    uint32_t base_row, scale_row, groups, k, M;
    uint32_t rows_per_cta, nbox;
    int x_dtype, y_dtype;
    uint32_t slot_bytes, nslots;
    uint32_t off_b, off_fo, off_red, off_bar;
    uint32_t *err;          // library error word
};

__device__ __forceinline__ float fp8_value(uint8_t b) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
}

__device__ __forceinline__ uint8_t to_fp8(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Issue the copies of tile `tile` into slot `slot` (called by a full warp):
// the tile's base rows as nbox tensor boxes of 32 rows x 128 bytes (128-byte
// swizzled; rows past the CTA's range are out of the map and come back zero
// without being read) and its scales as one 16-byte aligned bulk copy.
__device__ __forceinline__ void issue_tile(const Params &p, uint8_t *smem, uint64_t r_begin, uint64_t r_end,
                                           uint32_t slot, uint32_t tile, int lane, bool last_cta) {
    const uint64_t row0 = r_begin + (uint64_t)tile * kTile;
    const uint32_t nrows = r_end - row0 < (uint64_t)kTile ? (uint32_t)(r_end - row0) : (uint32_t)kTile;
    const uint8_t *s_src = p.scale + row0 * p.scale_row;
    const uintptr_t a = reinterpret_cast<uintptr_t>(s_src) & ~uintptr_t(15);
    const uintptr_t e = (reinterpret_cast<uintptr_t>(s_src) + (uintptr_t)nrows * p.scale_row + 15) & ~uintptr_t(15);
    const uint32_t s_bytes = (uint32_t)(e - a);
    const uint32_t bar = smem_u32(smem + p.off_bar) + 8 * slot;
    const uint32_t dst = smem_u32(smem) + slot * p.slot_bytes;
    if (lane == 0) mbar_arrive_expect_tx(bar, p.nbox * 4096u + s_bytes);
    __syncwarp();
    for (uint32_t bx = lane; bx < p.nbox; bx += 32) {
        if (last_cta)
            tma_load_2d(dst + bx * 4096u, &p.tmap_last, (int)(bx * 128), (int)(tile * kTile), bar);
        else
            tma_load_3d(dst + bx * 4096u, &p.tmap_main, (int)(bx * 128), (int)(tile * kTile), (int)blockIdx.x, bar);
    }
    if (lane == 0) bulk_g2s(dst + p.nbox * 4096u, reinterpret_cast<const void *>(a), s_bytes, bar);
}

// Swaps register-index bit R with lane bit L of a warp-held 32x32 array.
template <int R, int L>
__device__ __forceinline__ void swap_bits(float (&v)[32], int lane) {
    const bool a = (lane >> L) & 1;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        if (r & (1 << R)) continue;
        const float lo = v[r], hi = v[r | (1 << R)];
        const float recv = __shfl_xor_sync(0xffffffffu, a ? lo : hi, 1 << L);
        v[r] = a ? recv : lo;
        v[r | (1 << R)] = a ? hi : recv;
    }
}

// One halving step of a warp reduce-scatter over 2*HALF values per lane: lanes
// with bit log2(HALF) set keep the upper half, the others the lower half.
template <int HALF>
__device__ __forceinline__ void reduce_scatter_stage(float (&v)[32], int lane) {
    const bool hi = lane & HALF;
#pragma unroll
    for (int r = 0; r < HALF; ++r) {
        const float lo_v = v[r], hi_v = v[r + HALF];
        v[r] = (hi ? hi_v : lo_v) + __shfl_xor_sync(0xffffffffu, hi ? lo_v : hi_v, HALF);
    }
}

// Rotation of block `b` of token `m` and its three-term e4m3 B operand.
template <int NT>
__device__ __forceinline__ void prep_block(const Params &p, uint8_t *smem, uint32_t m, uint32_t b, int lane) {
    // natural layout: v[8*i + e] = element 256*i + 8*lane + e of the block
    float v[32];
    const uint64_t xrow = (uint64_t)m * p.k;
    const bool full = (b + 1) * 1024 <= p.k;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c = b * 1024 + 256 * i + 8 * lane;
        float t8[8];
        if (full) {
            load8(p.x, xrow + c, p.x_dtype, t8);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) t8[e] = c + e < p.k ? load1(p.x, xrow + c + e, p.x_dtype) : 0.f;
        }
        if (p.signs) {   // rotation implies k % 1024 == 0, so the block is full
            float d8[8];
            load_signs8(p.signs, c, d8);
#pragma unroll
            for (int e = 0; e < 8; ++e) t8[e] *= d8[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * i + e] = t8[e];
    }
    if (p.signs) {
        wht1024_warp(v, lane);
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] *= 0.03125f;
    }
    // element bits 0,1 go to lanes, 3,7 to registers: afterwards lane bits
    // (0..4) hold element bits (0,4,5,6,1) and register bits (0..4) hold
    // element bits (3,7,2,8,9)
    swap_bits<0, 0>(v, lane);
    swap_bits<1, 4>(v, lane);
    // within a group, B-fragment half h of quad lane t holds word t + 4h, i.e.
    // elements 64h + 16t + 4i + j: j = element bits 0,1, t = bits 4,5, h = bit 6
    const int j = (lane & 1) | ((lane >> 3) & 2);      // element bits 0,1
    const int t = (lane >> 1) & 3;                      // element bits 4,5
    const int h = (lane >> 3) & 1;                      // element bit 6
    float mx = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) mx = fmaxf(mx, fabsf(v[r]));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    int E = 0;
    if (mx > 0.f) E = 7 - ilogbf(mx);      // mx * 2^E in [128, 256)
    E = max(-120, min(120, E));
    const float up = __int_as_float((127 + E) << 23) * ((j & 1) ? 0.25f : 1.f);
    const float back = (j & 1) ? 4.f : 1.f;
    uint32_t *B = reinterpret_cast<uint32_t *>(smem + p.off_b);
    float sums[32];      // [3 * Gl + q], reduced over the warp below
#pragma unroll
    for (int Gl = 0; Gl < 8; ++Gl) {
        const uint32_t G = b * 8 + Gl;
        uint32_t w0 = 0, w1 = 0, w2 = 0;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = (i >> 1) | ((Gl & 1) << 1) | ((i & 1) << 2) | ((Gl >> 1) << 3);
            const float val = v[r] * up;
            const uint8_t c0 = to_fp8(val);
            const float f0 = fp8_value(c0);
            const float r1 = val - f0;
            const uint8_t c1 = to_fp8(r1 * 16.f);
            const float f1 = fp8_value(c1);
            const float r2 = r1 - f1 * 0.0625f;
            const uint8_t c2 = to_fp8(r2 * 256.f);
            const float f2 = fp8_value(c2);
            w0 |= (uint32_t)c0 << (8 * i);
            w1 |= (uint32_t)c1 << (8 * i);
            w2 |= (uint32_t)c2 << (8 * i);
            s0 += f0;
            s1 += f1;
            s2 += f2;
        }
        sums[3 * Gl] = s0 * back;
        sums[3 * Gl + 1] = s1 * back;
        sums[3 * Gl + 2] = s2 * back;
        if (G < p.groups) {
            const uint32_t words[3] = {w0, w1, w2};
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                const uint32_t col = 3 * m + q, T = col >> 3, gp = col & 7;
                B[((G * NT + T) * 4 + j) * 64 + (gp * 4 + t) * 2 + h] = words[q];
            }
        }
    }
    sums[24] = sums[25] = sums[26] = sums[27] = sums[28] = sums[29] = sums[30] = sums[31] = 0.f;
    // reduce-scatter: afterwards lane l holds the warp total of sums[l]
    reduce_scatter_stage<16>(sums, lane);
    reduce_scatter_stage<8>(sums, lane);
    reduce_scatter_stage<4>(sums, lane);
    reduce_scatter_stage<2>(sums, lane);
    reduce_scatter_stage<1>(sums, lane);
    // stage 2^s kept the upper half for lanes with bit s set, so lane l holds
    // the total of index l
    const int idx = lane;
    if (idx < 24) {
        const int Gl = idx / 3, q = idx % 3;
        const uint32_t G = b * 8 + Gl;
        if (G < p.groups) {
            const uint32_t col = 3 * m + q, T = col >> 3, gp = col & 7;
            float2 *FO = reinterpret_cast<float2 *>(smem + p.off_fo);
            FO[(G * NT + T) * 8 + gp] = make_float2(__int_as_float((127 + 9 - E - 4 * q) << 23),
                                                    sums[0] * __int_as_float((127 - E - 4 * q) << 23));
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(NT == 1 ? 512 : 256, 1) gemv_pq2_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = blockDim.x >> 5;
    const uint64_t r_begin = (uint64_t)blockIdx.x * p.rows_per_cta;
    const uint64_t r_end = r_begin + p.rows_per_cta < p.n ? r_begin + p.rows_per_cta : p.n;
    const bool last_cta = blockIdx.x == gridDim.x - 1;
    const uint32_t ntile = (uint32_t)((r_end - r_begin + kTile - 1) / kTile);
    const uint32_t bar0 = smem_u32(smem + p.off_bar);
    const uint32_t slot = warp >> 2, quarter = warp & 3;
    if (tid == 32) prefetch_tmap(last_cta ? &p.tmap_last : &p.tmap_main);

    if (tid == 0) {
        for (uint32_t s = 0; s < p.nslots; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // weights are read-only parameters: start streaming them before waiting on
    // the preceding kernel; one warp per slot issues its first tile
    if (quarter == 0 && slot < ntile) issue_tile(p, smem, r_begin, r_end, slot, slot, lane, last_cta);
    pdl_launch_dependents();

    {   // zero the B operand and its per-group factors (unused columns stay 0)
        uint4 *z = reinterpret_cast<uint4 *>(smem + p.off_b);
        const uint32_t nz = (p.off_red - p.off_b) / 16;
        for (uint32_t i = tid; i < nz; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    }
    pdl_wait();          // activations and the output belong to the preceding work
    __syncthreads();
    const uint32_t nblk = (p.k + 1023) / 1024;
    for (uint32_t task = warp; task < p.M * nblk; task += nwarps) prep_block<NT>(p, smem, task / nblk, task % nblk, lane);
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    const uint32_t g_lo = quarter * p.groups / 4, g_hi = (quarter + 1) * p.groups / 4;
    const uint32_t slot_addr = smem_u32(smem) + slot * p.slot_bytes;
    const uint32_t b_addr = smem_u32(smem + p.off_b), fo_addr = smem_u32(smem + p.off_fo);
    float *red = reinterpret_cast<float *>(smem + p.off_red) + slot * (2 * 3 * kTile * p.M);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t phase = 0;
    for (uint32_t tile = slot; tile < ntile; tile += p.nslots) {
        const uint64_t row0 = r_begin + (uint64_t)tile * kTile;
        const uint32_t nrows = r_end - row0 < (uint64_t)kTile ? (uint32_t)(r_end - row0) : (uint32_t)kTile;
        // a wait that runs out skips the tile's math but still meets the other
        // warps of the slot at the barrier, then all leave after one more wait
        const bool ready = mbar_wait(bar0 + 8 * slot, phase, p.err);
        phase ^= 1;
        const uint32_t s_delta = (uint32_t)(reinterpret_cast<uintptr_t>(p.scale + row0 * p.scale_row) & 15);
        const uint32_t sc_addr = slot_addr + p.nbox * 4096u + s_delta;

        float acc[2][NT][4];
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int T = 0; T < NT; ++T)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[rb][T][i] = 0.f;

        // software pipeline: the next group's weight words and scales are
        // requested before the current group's MMAs
        uint32_t wn[2][4];
        uint32_t sn[2][2];
        // word w of group G of tile row r sits in box G/4 at
        // r*128 + (((G % 4) * 2 + w / 4) ^ (r % 8)) * 16 + (w % 4) * 4;
        // lane (g, t) reads words t and t + 4 of rows g (+8, +16, +24):
        // eight rows hit eight different 16-byte chunks, so no bank conflicts
        const uint32_t row_base = slot_addr + g * 128 + 4 * t;
        auto fetch = [&](uint32_t G, uint32_t (&w)[2][4], uint32_t (&sv)[2][2]) {
            const uint32_t gb = row_base + (G >> 2) * 4096u;
            const uint32_t c0 = (((G & 3) * 2) ^ g) * 16, c1 = (((G & 3) * 2 + 1) ^ g) * 16;
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                const uint32_t rr = gb + rb * 2048;
                w[rb][0] = lds32(rr + c0);          // row g,   word t
                w[rb][1] = lds32(rr + c1);          // row g,   word t + 4
                w[rb][2] = lds32(rr + 1024 + c0);   // row g+8, word t
                w[rb][3] = lds32(rr + 1024 + c1);   // row g+8, word t + 4
                sv[rb][0] = lds16(sc_addr + (16 * rb + g) * p.scale_row + 2 * G);
                sv[rb][1] = lds16(sc_addr + (16 * rb + g + 8) * p.scale_row + 2 * G);
            }
        };
        if (ready && g_lo < g_hi) fetch(g_lo, wn, sn);
        for (uint32_t G = g_lo; ready && G < g_hi; ++G) {
            uint32_t w[2][4], sv[2][2];
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
#pragma unroll
                for (int i = 0; i < 4; ++i) w[rb][i] = wn[rb][i];
                sv[rb][0] = sn[rb][0];
                sv[rb][1] = sn[rb][1];
            }
            if (G + 1 < g_hi) fetch(G + 1, wn, sn);
            float d[2][NT][4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t mask = (jj & 1) ? 0x0C0C0C0Cu : 0x03030303u;
                const int sh = (jj & 2) ? 4 : 0;
                uint32_t a[2][4];
#pragma unroll
                for (int rb = 0; rb < 2; ++rb) {
                    a[rb][0] = (w[rb][0] >> sh) & mask;   // row g,   k-slots 4t..4t+3   <- word t
                    a[rb][1] = (w[rb][2] >> sh) & mask;   // row g+8, k-slots 4t..4t+3   <- word t
                    a[rb][2] = (w[rb][1] >> sh) & mask;   // row g,   k-slots 16+4t..    <- word t+4
                    a[rb][3] = (w[rb][3] >> sh) & mask;   // row g+8, k-slots 16+4t..    <- word t+4
                }
#pragma unroll
                for (int T = 0; T < NT; ++T) {
                    const uint2 bf = lds64(b_addr + (((G * NT + T) * 4 + jj) * 64 + lane * 2) * 4);
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        if (jj == 0) mma_e4m3(d[rb][T], a[rb], bf.x, bf.y, zero4);
                        else mma_e4m3(d[rb][T], a[rb], bf.x, bf.y, d[rb][T]);
                    }
                }
            }
            float sr[2][2];
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                sr[rb][0] = __half2float(__ushort_as_half((unsigned short)sv[rb][0]));
                sr[rb][1] = __half2float(__ushort_as_half((unsigned short)sv[rb][1]));
            }
#pragma unroll
            for (int T = 0; T < NT; ++T) {
                const float4 fo = lds128f(fo_addr + ((G * NT + T) * 8 + 2 * t) * 8);
#pragma unroll
                for (int rb = 0; rb < 2; ++rb) {
                    acc[rb][T][0] = fmaf(sr[rb][0], fmaf(fo.x, d[rb][T][0], -fo.y), acc[rb][T][0]);
                    acc[rb][T][1] = fmaf(sr[rb][0], fmaf(fo.z, d[rb][T][1], -fo.w), acc[rb][T][1]);
                    acc[rb][T][2] = fmaf(sr[rb][1], fmaf(fo.x, d[rb][T][2], -fo.y), acc[rb][T][2]);
                    acc[rb][T][3] = fmaf(sr[rb][1], fmaf(fo.z, d[rb][T][3], -fo.w), acc[rb][T][3]);
                }
            }
        }

        // gather the three term columns of each token inside the quad
        float yp[2][2][2];     // [rb][row g / g+8][token t / t+4]
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int rs = 0; rs < 2; ++rs) {
                float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
                for (int T = 0; T < NT; ++T)
#pragma unroll
                    for (int par = 0; par < 2; ++par)
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt) {
                            const float val = __shfl_sync(0xffffffffu, acc[rb][T][2 * rs + par], (lane & ~3) | tt);
                            const int tok = (8 * T + 2 * tt + par) / 3;
                            if (tok == t) s_lo += val;
                            else if (tok == t + 4) s_hi += val;
                        }
                yp[rb][rs][0] = s_lo;
                yp[rb][rs][1] = s_hi;
            }
        // reduce the four k-quarters of the slot: [buf][quarter-1][token][row]
        float *rbuf = red + ((tile / p.nslots) & 1) * (3 * kTile * p.M);
        if (quarter) {
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                for (int rs = 0; rs < 2; ++rs) {
                    const int rl = 16 * rb + 8 * rs + g;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t m = t + 4 * u;
                        if (m < p.M) rbuf[((quarter - 1) * p.M + m) * kTile + rl] = yp[rb][rs][u];
                    }
                }
        }
        named_barrier(1 + slot, 128);
        if (!ready) {
            mbar_wait(bar0 + 8 * slot, phase ^ 1, p.err);
            return;
        }
        if (!quarter) {
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                for (int rs = 0; rs < 2; ++rs) {
                    const uint32_t rl = 16 * rb + 8 * rs + g;
                    if (rl >= nrows) continue;
                    const uint64_t r = row0 + rl;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t m = t + 4 * u;
                        if (m < p.M) {
                            const float tot = yp[rb][rs][u] + rbuf[(0 * p.M + m) * kTile + rl] +
                                              rbuf[(1 * p.M + m) * kTile + rl] + rbuf[(2 * p.M + m) * kTile + rl];
                            store1(p.y, (uint64_t)m * p.n + r, p.y_dtype, tot);
                        }
                    }
                }
            if (tile + p.nslots < ntile) {
                fence_proxy_async();
                issue_tile(p, smem, r_begin, r_end, slot, tile + p.nslots, lane, last_cta);
            }
        }
    }
}

}  // namespace

bool gemv_pq2_plan(const ninfer_row_split_geometry &g, uint64_t M, bool rotate, int sms, int smem_limit,
                   GemvPlan *plan) {
    *plan = GemvPlan{};
    if (M < 2 || M > 8) return false;
    if (rotate && g.k % 1024) return false;
    if (g.payload_bytes % 16 || g.base_row_bytes % 16) return false;
    if (g.k > (1u << 24) || g.groups_per_row > (1u << 16) || g.n > (1ull << 31)) return false;
    const uint32_t NT = (uint32_t)((3 * M + 7) / 8);
    const uint32_t groups = (uint32_t)g.groups_per_row;
    const uint32_t nbox = (uint32_t)((g.base_row_bytes + 127) / 128);
    const uint32_t scale_area = ((kTile * (uint32_t)g.scale_row_bytes + 16 + 15) / 16) * 16;
    const uint32_t slot_bytes = ((nbox * 4096u + scale_area + 1023) / 1024) * 1024;
    const uint32_t b_bytes = groups * NT * 1024;
    const uint32_t fo_bytes = groups * NT * 64;
    const uint32_t red_bytes = kMaxSlots * 2 * 3 * kTile * (uint32_t)M * 4;
    const uint32_t bar_bytes = 64;
    // rows per CTA: ceil(n / grid) for all CTAs but the last
    const uint64_t grid0 = std::min<uint64_t>((uint64_t)sms, (g.n + kTile - 1) / kTile);
    const uint64_t R = (g.n + grid0 - 1) / grid0;
    const uint64_t grid = (g.n + R - 1) / R;
    const uint64_t tiles = (R + kTile - 1) / kTile;
    const uint64_t fixed = (uint64_t)b_bytes + fo_bytes + red_bytes + bar_bytes;
    if (fixed + slot_bytes > (uint64_t)smem_limit) return false;
    const uint64_t max_slots = NT == 1 ? kMaxSlots : kMaxSlots / 2;     // 4 warps per slot, register budget
    const uint32_t nslots = (uint32_t)std::min<uint64_t>({max_slots, tiles, ((uint64_t)smem_limit - fixed) / slot_bytes});
    if (nslots == 0) return false;
    plan->ok = true;
    plan->grid = (uint32_t)grid;
    plan->rows_per_cta = (uint32_t)R;
    plan->nbox = nbox;
    plan->nt = NT;
    plan->nslots = nslots;
    plan->slot_bytes = slot_bytes;
    plan->off_b = nslots * slot_bytes;
    plan->off_fo = plan->off_b + b_bytes;
    plan->off_red = plan->off_fo + fo_bytes;
    plan->off_bar = plan->off_red + red_bytes;
    plan->smem = plan->off_bar + bar_bytes;
    return true;
}


int gemv_pq2_launch(const GemvPlan &plan, const uint8_t *payload, const ninfer_row_split_geometry &g, const void *x,
                    int x_dtype, const uint16_t *signs, void *y, int y_dtype, uint64_t M, cudaStream_t stream,
                    bool pdl) {
    Params p;
    std::memset(&p, 0, sizeof p);
    p.base = payload + g.base_offset;
    p.scale = payload + g.scale_offset;
    p.x = x;
    p.signs = signs;
    p.y = y;
    p.n = g.n;
    p.base_row = (uint32_t)g.base_row_bytes;
    p.scale_row = (uint32_t)g.scale_row_bytes;
    p.groups = (uint32_t)g.groups_per_row;
    p.k = (uint32_t)g.k;
    p.M = (uint32_t)M;
    p.rows_per_cta = plan.rows_per_cta;
    p.nbox = plan.nbox;
    p.x_dtype = x_dtype;
    p.y_dtype = y_dtype;
    p.slot_bytes = plan.slot_bytes;
    p.nslots = plan.nslots;
    p.off_b = plan.off_b;
    p.off_fo = plan.off_fo;
    p.off_red = plan.off_red;
    p.off_bar = plan.off_bar;
    int st = device_error_word(&p.err);
    if (st) return st;
    const uint64_t R = plan.rows_per_cta, G = plan.grid;
    if (G > 1) {
        st = encode_rows(&p.tmap_main, p.base, g.base_row_bytes, R, G - 1, 128, kTile, true);
        if (st) return st;
    }
    st = encode_rows(&p.tmap_last, p.base + (G - 1) * R * g.base_row_bytes, g.base_row_bytes, g.n - (G - 1) * R, 1, 128, kTile, true);
    if (st) return st;
    void (*kern)(const Params) = plan.nt == 1 ? gemv_pq2_kernel<1> : plan.nt == 2 ? gemv_pq2_kernel<2> : gemv_pq2_kernel<3>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv: smem attribute: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.nslots * 4 * 32);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return fail(NINFER_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    return NINFER_OK;
}

}  // namespace ninfer

