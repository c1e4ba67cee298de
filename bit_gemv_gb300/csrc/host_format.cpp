// Host side of the boundary: status strings, the row-split plane geometry, the
// plane packer/unpacker and the ggml block <-> plane conversion.
//
// Sources: "bonsai三元GGUF模型转ninfer模型01" (ninfer ternary artifact format page)
// §2 (TernaryFormat PQ2_0_G128 = (128, 32, 0), PTQ1_0_G128 = (128, 24, 2)),
// §3 (row_split_geometry, plane order vs block byte order), §4 (GGML_BLOCK,
// BLOCK_PLANE_SLICES); "GGUF 完整讲解" §4.3 (Q2_0 2-bit fields, least
// significant first, value = code - 1).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <thread>
#include <vector>

#include "common.h"

namespace ninfer {

static thread_local std::string t_last_error;

int fail(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

void clear_error() { t_last_error.clear(); }

static const FormatInfo kFormats[] = {
    {NINFER_PQ2_0_G128, "PQ2_0_G128", 128, 32, 0, 34},
    {NINFER_PTQ1_0_G128, "PTQ1_0_G128", 128, 24, 2, 28},
};

const FormatInfo *format_info(int fmt) {
    for (const auto &f : kFormats)
        if (f.id == fmt) return &f;
    return nullptr;
}

static inline bool align_up_ok(uint64_t v, uint64_t a, uint64_t *out) {
    uint64_t t;
    if (!add_ok(v, a - 1, &t)) return false;
    *out = t / a * a;
    return true;
}

int geometry(int fmt, uint64_t n, uint64_t k, ninfer_row_split_geometry *g) {
    const FormatInfo *f = format_info(fmt);
    if (!f) return fail(NINFER_ERR_UNKNOWN_FORMAT, "unknown numeric format id %d (expected 142 PQ2_0_G128 or 143 PTQ1_0_G128)", fmt);
    if (n == 0 || k == 0) return fail(NINFER_ERR_SHAPE, "shape must have positive dimensions (n=%llu, k=%llu)",
                                      (unsigned long long)n, (unsigned long long)k);
    ninfer_row_split_geometry r{};
    r.n = n;
    r.k = k;
    bool ok = align_up_ok(k, f->group, &r.k_pad);
    r.groups_per_row = ok ? r.k_pad / f->group : 0;
    r.base_bytes_per_group = f->base_bytes;
    r.high_bytes_per_group = f->high_bytes;
    ok = ok && mul_ok(r.groups_per_row, f->base_bytes, &r.base_row_bytes);
    ok = ok && mul_ok(r.groups_per_row, f->high_bytes, &r.high_row_bytes);
    ok = ok && mul_ok(r.groups_per_row, 2, &r.scale_row_bytes);
    r.base_offset = 0;
    ok = ok && mul_ok(n, r.base_row_bytes, &r.base_bytes);
    ok = ok && align_up_ok(r.base_offset + r.base_bytes, 256, &r.high_offset);
    ok = ok && mul_ok(n, r.high_row_bytes, &r.high_bytes);
    uint64_t high_span = 0;
    ok = ok && align_up_ok(r.high_bytes, 256, &high_span);
    ok = ok && add_ok(r.high_offset, high_span, &r.scale_offset);
    ok = ok && mul_ok(n, r.scale_row_bytes, &r.scale_bytes);
    ok = ok && add_ok(r.scale_offset, r.scale_bytes, &r.payload_bytes);
    if (!ok) return fail(NINFER_ERR_OVERFLOW, "geometry of (%llu, %llu) overflows 64 bits",
                         (unsigned long long)n, (unsigned long long)k);
    *g = r;
    return NINFER_OK;
}

// Runs fn(row_begin, row_end) over [0, n) on up to hardware_concurrency threads.
template <class Fn>
static void parallel_rows(uint64_t n, uint64_t work_per_row, Fn fn) {
    unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    uint64_t total = n * std::max<uint64_t>(work_per_row, 1);
    unsigned nt = total < (1u << 22) ? 1u : std::min<unsigned>(hw, 32u);
    nt = (unsigned)std::min<uint64_t>(nt, n);
    if (nt <= 1) {
        fn(0, n);
        return;
    }
    std::vector<std::thread> th;
    for (unsigned t = 0; t < nt; ++t) {
        uint64_t b = n * t / nt, e = n * (t + 1) / nt;
        th.emplace_back([=] { fn(b, e); });
    }
    for (auto &x : th) x.join();
}

}  // namespace ninfer

using namespace ninfer;

extern "C" {

const char *ninfer_last_error(void) { return t_last_error.c_str(); }

int ninfer_abi_version(void) { return NINFER_TERNARY_ABI_VERSION; }

const char *ninfer_status_name(int s) {
    switch (s) {
        case NINFER_OK: return "NINFER_OK";
        case NINFER_ERR_INVALID_ARGUMENT: return "NINFER_ERR_INVALID_ARGUMENT";
        case NINFER_ERR_UNKNOWN_FORMAT: return "NINFER_ERR_UNKNOWN_FORMAT";
        case NINFER_ERR_SHAPE: return "NINFER_ERR_SHAPE";
        case NINFER_ERR_SIZE_MISMATCH: return "NINFER_ERR_SIZE_MISMATCH";
        case NINFER_ERR_ALIGNMENT: return "NINFER_ERR_ALIGNMENT";
        case NINFER_ERR_INVALID_CODE: return "NINFER_ERR_INVALID_CODE";
        case NINFER_ERR_CUDA: return "NINFER_ERR_CUDA";
        case NINFER_ERR_OVERFLOW: return "NINFER_ERR_OVERFLOW";
        default: return "NINFER_ERR_UNKNOWN_STATUS";
    }
}

int ninfer_ternary_geometry(int fmt, uint64_t n, uint64_t k, ninfer_row_split_geometry *out) {
    if (!out) return fail(NINFER_ERR_INVALID_ARGUMENT, "geometry output pointer is NULL");
    return geometry(fmt, n, k, out);
}

int ninfer_ternary_pack(int fmt, uint64_t n, uint64_t k, const int8_t *values,
                        const uint16_t *scales_f16, uint8_t *payload, uint64_t payload_bytes) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!values || !scales_f16 || !payload) return fail(NINFER_ERR_INVALID_ARGUMENT, "pack: NULL buffer");
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    // validate values first so a failure writes nothing
    std::atomic<uint64_t> bad{UINT64_MAX};
    parallel_rows(n, k, [&](uint64_t r0, uint64_t r1) {
        for (uint64_t r = r0; r < r1; ++r) {
            const int8_t *v = values + r * k;
            for (uint64_t c = 0; c < k; ++c)
                if (v[c] < -1 || v[c] > 1) {
                    uint64_t idx = r * k + c, cur = bad.load();
                    while (idx < cur && !bad.compare_exchange_weak(cur, idx)) {}
                    break;
                }
        }
    });
    if (bad.load() != UINT64_MAX)
        return fail(NINFER_ERR_INVALID_CODE, "value at flat index %llu is not -1, 0 or +1",
                    (unsigned long long)bad.load());
    std::memset(payload, 0, payload_bytes);
    const uint64_t G = g.groups_per_row;
    parallel_rows(n, k, [&](uint64_t r0, uint64_t r1) {
        uint8_t codes[128];
        for (uint64_t r = r0; r < r1; ++r) {
            const int8_t *v = values + r * k;
            uint8_t *base = payload + g.base_offset + r * g.base_row_bytes;
            uint8_t *high = payload + g.high_offset + r * g.high_row_bytes;
            for (uint64_t gi = 0; gi < G; ++gi) {
                for (uint64_t j = 0; j < 128; ++j) {
                    uint64_t c = gi * 128 + j;
                    codes[j] = (uint8_t)((c < k ? v[c] : 0) + 1);  // pad weights: value 0
                }
                if (fmt == NINFER_PQ2_0_G128) {
                    uint8_t *b = base + gi * 32;
                    for (int j = 0; j < 32; ++j)
                        b[j] = (uint8_t)(codes[4 * j] | (codes[4 * j + 1] << 2) | (codes[4 * j + 2] << 4) |
                                         (codes[4 * j + 3] << 6));
                } else {
                    uint8_t *b = base + gi * 24;
                    for (int j = 0; j < 24; ++j) {
                        const uint8_t *t = codes + 5 * j;
                        b[j] = (uint8_t)(t[0] + 3 * t[1] + 9 * t[2] + 27 * t[3] + 81 * t[4]);
                    }
                    uint8_t *h = high + gi * 2;
                    for (int j = 0; j < 2; ++j) {
                        const uint8_t *t = codes + 120 + 4 * j;
                        h[j] = (uint8_t)(t[0] + 3 * t[1] + 9 * t[2] + 27 * t[3]);
                    }
                }
            }
            uint8_t *s = payload + g.scale_offset + r * g.scale_row_bytes;
            for (uint64_t gi = 0; gi < G; ++gi) {
                uint16_t w = scales_f16[r * G + gi];
                s[2 * gi] = (uint8_t)(w & 0xff);
                s[2 * gi + 1] = (uint8_t)(w >> 8);
            }
        }
    });
    return NINFER_OK;
}

int ninfer_ternary_unpack(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                          uint64_t payload_bytes, int8_t *values, uint16_t *scales_f16) {
    ninfer_row_split_geometry g;
    int st = geometry(fmt, n, k, &g);
    if (st) return st;
    if (!values || !scales_f16 || !payload) return fail(NINFER_ERR_INVALID_ARGUMENT, "unpack: NULL buffer");
    if (payload_bytes != g.payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g.payload_bytes);
    const uint64_t G = g.groups_per_row;
    std::atomic<uint64_t> bad{UINT64_MAX};
    parallel_rows(n, k, [&](uint64_t r0, uint64_t r1) {
        int8_t vals[128];
        for (uint64_t r = r0; r < r1; ++r) {
            const uint8_t *base = payload + g.base_offset + r * g.base_row_bytes;
            const uint8_t *high = payload + g.high_offset + r * g.high_row_bytes;
            for (uint64_t gi = 0; gi < G; ++gi) {
                bool invalid = false;
                if (fmt == NINFER_PQ2_0_G128) {
                    const uint8_t *b = base + gi * 32;
                    for (int j = 0; j < 128; ++j) {
                        int code = (b[j >> 2] >> (2 * (j & 3))) & 3;
                        invalid |= code == 3;
                        vals[j] = (int8_t)(code - 1);
                    }
                } else {
                    const uint8_t *b = base + gi * 24;
                    for (int j = 0; j < 24; ++j) {
                        int byte = b[j];
                        invalid |= byte >= 243;
                        for (int i = 0; i < 5; ++i) { vals[5 * j + i] = (int8_t)(byte % 3 - 1); byte /= 3; }
                    }
                    const uint8_t *h = high + gi * 2;
                    for (int j = 0; j < 2; ++j) {
                        int byte = h[j];
                        invalid |= byte >= 81;
                        for (int i = 0; i < 4; ++i) { vals[120 + 4 * j + i] = (int8_t)(byte % 3 - 1); byte /= 3; }
                    }
                }
                if (invalid) {
                    uint64_t idx = r * G + gi, cur = bad.load();
                    while (idx < cur && !bad.compare_exchange_weak(cur, idx)) {}
                }
                for (uint64_t j = 0; j < 128; ++j) {
                    uint64_t c = gi * 128 + j;
                    if (c < k) values[r * k + c] = vals[j];
                }
            }
            const uint8_t *s = payload + g.scale_offset + r * g.scale_row_bytes;
            for (uint64_t gi = 0; gi < G; ++gi)
                scales_f16[r * G + gi] = (uint16_t)(s[2 * gi] | (s[2 * gi + 1] << 8));
        }
    });
    if (bad.load() != UINT64_MAX) {
        uint64_t idx = bad.load();
        return fail(NINFER_ERR_INVALID_CODE, "row %llu group %llu holds a code no ternary value packs to",
                    (unsigned long long)(idx / G), (unsigned long long)(idx % G));
    }
    return NINFER_OK;
}

// BLOCK_PLANE_SLICES of the format page §4: (start, length) of base, high, scale.
static void block_slices(int fmt, int *bs, int *bl, int *hs, int *hl, int *ss) {
    if (fmt == NINFER_PQ2_0_G128) { *bs = 2; *bl = 32; *hs = 0; *hl = 0; *ss = 0; }
    else { *bs = 0; *bl = 24; *hs = 24; *hl = 2; *ss = 26; }
}

static int blocks_check(int fmt, uint64_t n, uint64_t k, const void *a, const void *b,
                        uint64_t blocks_bytes, uint64_t payload_bytes, ninfer_row_split_geometry *g) {
    int st = geometry(fmt, n, k, g);
    if (st) return st;
    if (!a || !b) return fail(NINFER_ERR_INVALID_ARGUMENT, "block conversion: NULL buffer");
    const FormatInfo *f = format_info(fmt);
    uint64_t want;
    if (!mul_ok(n * g->groups_per_row, f->block_bytes, &want))
        return fail(NINFER_ERR_OVERFLOW, "block stream size overflows");
    if (blocks_bytes != want)
        return fail(NINFER_ERR_SIZE_MISMATCH, "block stream holds %llu bytes; shape requires %llu",
                    (unsigned long long)blocks_bytes, (unsigned long long)want);
    if (payload_bytes != g->payload_bytes)
        return fail(NINFER_ERR_SIZE_MISMATCH, "payload stores %llu bytes; layout requires %llu",
                    (unsigned long long)payload_bytes, (unsigned long long)g->payload_bytes);
    return NINFER_OK;
}

int ninfer_blocks_to_planes(int fmt, uint64_t n, uint64_t k, const uint8_t *blocks,
                            uint64_t blocks_bytes, uint8_t *payload, uint64_t payload_bytes) {
    ninfer_row_split_geometry g;
    int st = blocks_check(fmt, n, k, blocks, payload, blocks_bytes, payload_bytes, &g);
    if (st) return st;
    int bs, bl, hs, hl, ss;
    block_slices(fmt, &bs, &bl, &hs, &hl, &ss);
    const uint64_t nb = format_info(fmt)->block_bytes, G = g.groups_per_row;
    std::memset(payload, 0, payload_bytes);
    parallel_rows(n, g.k_pad, [&](uint64_t r0, uint64_t r1) {
        for (uint64_t r = r0; r < r1; ++r)
            for (uint64_t gi = 0; gi < G; ++gi) {
                const uint8_t *blk = blocks + (r * G + gi) * nb;
                std::memcpy(payload + g.base_offset + r * g.base_row_bytes + gi * bl, blk + bs, bl);
                if (hl) std::memcpy(payload + g.high_offset + r * g.high_row_bytes + gi * hl, blk + hs, hl);
                std::memcpy(payload + g.scale_offset + r * g.scale_row_bytes + gi * 2, blk + ss, 2);
            }
    });
    return NINFER_OK;
}

int ninfer_planes_to_blocks(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                            uint64_t payload_bytes, uint8_t *blocks, uint64_t blocks_bytes) {
    ninfer_row_split_geometry g;
    int st = blocks_check(fmt, n, k, blocks, payload, blocks_bytes, payload_bytes, &g);
    if (st) return st;
    int bs, bl, hs, hl, ss;
    block_slices(fmt, &bs, &bl, &hs, &hl, &ss);
    const uint64_t nb = format_info(fmt)->block_bytes, G = g.groups_per_row;
    parallel_rows(n, g.k_pad, [&](uint64_t r0, uint64_t r1) {
        for (uint64_t r = r0; r < r1; ++r)
            for (uint64_t gi = 0; gi < G; ++gi) {
                uint8_t *blk = blocks + (r * G + gi) * nb;
                std::memcpy(blk + bs, payload + g.base_offset + r * g.base_row_bytes + gi * bl, bl);
                if (hl) std::memcpy(blk + hs, payload + g.high_offset + r * g.high_row_bytes + gi * hl, hl);
                std::memcpy(blk + ss, payload + g.scale_offset + r * g.scale_row_bytes + gi * 2, 2);
            }
    });
    return NINFER_OK;
}

}  // extern "C"

extern "C" int ninfer_validate_signs(const uint16_t *signs_bf16, uint64_t K) {
    using namespace ninfer;
    if (!signs_bf16) return fail(NINFER_ERR_INVALID_ARGUMENT, "validate signs: NULL vector");
    if (K == 0 || K % 1024)
        return fail(NINFER_ERR_SHAPE, "validate signs: K=%llu is not a positive multiple of 1024", (unsigned long long)K);
    for (uint64_t i = 0; i < K; ++i)
        if (signs_bf16[i] != 0x3F80u && signs_bf16[i] != 0xBF80u)
            return fail(NINFER_ERR_INVALID_ARGUMENT, "validate signs: entry %llu is 0x%04x, not +1 (0x3F80) or -1 (0xBF80)",
                        (unsigned long long)i, (unsigned)signs_bf16[i]);
    return NINFER_OK;
}
