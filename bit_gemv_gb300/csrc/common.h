// Internal helpers shared by the library's translation units: status/last-error
// handling, overflow-checked size arithmetic and the plane geometry.
#pragma once

#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "ninfer_ternary.h"

namespace ninfer {

// Records a formatted message as this thread's last error and returns status.
int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

inline bool mul_ok(uint64_t a, uint64_t b, uint64_t *out) { return !__builtin_mul_overflow(a, b, out); }
inline bool add_ok(uint64_t a, uint64_t b, uint64_t *out) { return !__builtin_add_overflow(a, b, out); }

struct FormatInfo {
    int id;
    const char *name;
    uint64_t group;       // weights per group
    uint64_t base_bytes;  // per group
    uint64_t high_bytes;  // per group
    uint64_t block_bytes; // ggml single-group block
};

// Returns nullptr for an unknown format id.
const FormatInfo *format_info(int fmt);

// row_split_geometry of the format page §3; returns a status (sets last error).
int geometry(int fmt, uint64_t n, uint64_t k, ninfer_row_split_geometry *g);

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace ninfer
