/*
 * ninfer_ternary.h -- C ABI of the GB300 (sm_103a) Hadamard-rotated ternary
 * projection library (libninfer_ternary.so).
 *
 * The library computes y = W . T(x): activations x (M x k) are rotated by the
 * signed block Walsh-Hadamard transform T(x) = H(D.x)/sqrt(1024) per 1024-wide
 * block, and multiplied by ternary weights W (n x k) stored in the row-split
 * PQ2_0_G128 / PTQ1_0_G128 plane layout. It also provides the inverse transform
 * for embedding rows, the host-side plane geometry and plane packers.
 *
 * Sources (web pages; cited by title and section):
 *   [FMT]  "bonsai三元GGUF模型转ninfer模型01" -- ninfer ternary artifact format
 *          page: §2 ternary numeric formats, §3 row-split plane geometry,
 *          §4 block <-> plane conversion, §6 constants.
 *   [GGUF] "GGUF 完整讲解" -- §4.3 the Q2_0 dequantisation (2-bit field order,
 *          offset code -> value).
 *   [V3]   NInfer "artifact-container.md" -- §6.1 numeric formats, §6.2 layouts
 *          (256-byte object alignment), §8 the hadamard_signs auxiliary,
 *          §11.3 / §12.6 error ownership ("refuse rather than run wrong").
 *   [TS]   "从 TensorSharp 视角解读 Ternary Bonsai 2 27B" -- §4.2 transform
 *          contract, §4.4 where the transforms apply.
 *
 * Conventions shared by every entry point
 *   - Sizes are uint64_t element or byte counts; data is little-endian.
 *   - Every function returns an ninfer_status. NINFER_OK is 0. On any other
 *     status nothing was launched or written, and ninfer_last_error() returns a
 *     thread-local message naming the argument at fault.
 *   - Host pointers ("host") are read/written synchronously. Device pointers
 *     ("device") must be device (or managed) memory the caller allocated and
 *     owns; the library never frees or retains them, and performs all device
 *     work asynchronously on the given stream (a cudaStream_t; NULL = the
 *     legacy default stream). Device pointers must be 16-byte aligned; packed
 *     weight payloads 256-byte aligned (the plane alignment of [FMT] §1 and
 *     [V3] §6.2).
 *   - The library allocates no device memory in any call. Kernels never trap
 *     or assert; device-side input problems are reported through an optional
 *     caller-owned status word.
 */
#ifndef NINFER_TERNARY_H
#define NINFER_TERNARY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NINFER_TERNARY_ABI_VERSION 1

/* Numeric formats ([FMT] §2, GGUF type ids from [FMT] §6 / [TS] §4.1). */
typedef enum {
    NINFER_PQ2_0_G128 = 142,  /* 32 base bytes + 2 scale bytes per 128 weights */
    NINFER_PTQ1_0_G128 = 143  /* 24 base + 2 high + 2 scale bytes per 128 weights */
} ninfer_format;

/* Element types of activations / outputs. */
typedef enum {
    NINFER_F32 = 0,
    NINFER_BF16 = 1,
    NINFER_F16 = 2
} ninfer_dtype;

typedef enum {
    NINFER_OK = 0,
    NINFER_ERR_INVALID_ARGUMENT = 1, /* null pointer, zero size, bad enum value */
    NINFER_ERR_UNKNOWN_FORMAT = 2,   /* format id is not 142 / 143 */
    NINFER_ERR_SHAPE = 3,            /* shape violates a rule (e.g. k % 1024 with signs) */
    NINFER_ERR_SIZE_MISMATCH = 4,    /* buffer size != the size the layout requires */
    NINFER_ERR_ALIGNMENT = 5,        /* pointer not aligned as required */
    NINFER_ERR_INVALID_CODE = 6,     /* packed bytes hold no ternary value */
    NINFER_ERR_CUDA = 7,             /* a CUDA runtime call failed (message has it) */
    NINFER_ERR_OVERFLOW = 8          /* a size does not fit in 64 bits */
} ninfer_status;

/* cudaStream_t without including CUDA headers. */
typedef struct CUstream_st *ninfer_stream;

/*
 * RowSplitGeometry: the 16 fields of row_split_geometry(format, shape), in the
 * page's order ([FMT] §3):
 *   k_pad = align_up(k, 128); groups_per_row = k_pad / 128;
 *   *_row_bytes = groups_per_row * per-group bytes (scale: 2, one binary16);
 *   base_offset = 0; high_offset = align_up(base_bytes, 256) (computed even
 *   when high_bytes == 0, so PQ2_0 has scale_offset == high_offset);
 *   scale_offset = high_offset + align_up(high_bytes, 256);
 *   payload_bytes = scale_offset + scale_bytes;
 *   plane sizes are n * the per-row sizes.
 * Planes are row-major [row][group][bytes].
 */
typedef struct {
    uint64_t n, k, k_pad, groups_per_row;
    uint64_t base_bytes_per_group, high_bytes_per_group;
    uint64_t base_row_bytes, high_row_bytes, scale_row_bytes;
    uint64_t base_offset, base_bytes;
    uint64_t high_offset, high_bytes;
    uint64_t scale_offset, scale_bytes;
    uint64_t payload_bytes;
} ninfer_row_split_geometry;

/* Thread-local description of the last non-OK status returned on this thread. */
const char *ninfer_last_error(void);
/* Static name of a status value ("NINFER_OK", ...). */
const char *ninfer_status_name(int status);
/* NINFER_TERNARY_ABI_VERSION of the loaded library. */
int ninfer_abi_version(void);

/*
 * ninfer_ternary_geometry -- [FMT] §3 row_split_geometry.
 *   fmt: ninfer_format; n, k: output rows and input width, both > 0.
 *   out: host struct, written on success.
 * Errors: UNKNOWN_FORMAT, SHAPE (n or k == 0), OVERFLOW, INVALID_ARGUMENT (out NULL).
 */
int ninfer_ternary_geometry(int fmt, uint64_t n, uint64_t k,
                            ninfer_row_split_geometry *out);

/*
 * ninfer_ternary_pack -- ternary values + group scales -> row-split payload (host).
 *   values: host int8[n * k], row-major, each -1, 0 or +1.
 *   scales_f16: host uint16[n * groups_per_row], binary16 bit patterns, one per
 *     128-weight group ([FMT] §3: "one binary16 per group").
 *   payload: host uint8[payload_bytes] written completely (pad bytes included).
 * Encoding (value v, code c = v + 1):
 *   PQ2_0_G128: group byte j holds weights 4j..4j+3, weight i in bits
 *     2*(i % 4) (least significant field first) -- the Q2_0 layout of
 *     [GGUF] §4.3, where code c decodes to c - 1.
 *   PTQ1_0_G128: base byte b (0..23) = sum_{i<5} c[5b+i] * 3^i, high byte h
 *     (0..1) = sum_{i<4} c[120+4h+i] * 3^i (little-endian base-3 digits; the
 *     pages fix 24 + 2 bytes per 128 weights but no digit order).
 *   Pad weights (columns k..k_pad-1) encode value 0.
 * Errors: UNKNOWN_FORMAT, SHAPE, INVALID_ARGUMENT, SIZE_MISMATCH (payload_bytes
 *   != geometry.payload_bytes), INVALID_CODE (a value outside {-1,0,+1}).
 */
int ninfer_ternary_pack(int fmt, uint64_t n, uint64_t k, const int8_t *values,
                        const uint16_t *scales_f16, uint8_t *payload,
                        uint64_t payload_bytes);

/*
 * ninfer_ternary_unpack -- exact inverse of ninfer_ternary_pack (host).
 *   values: host int8[n * k] out; scales_f16: host uint16[n * groups_per_row] out.
 * Errors: as pack, plus INVALID_CODE when a PQ2_0 field holds code 3 or a
 *   PTQ1_0 base byte is >= 243 / high byte >= 81 (no ternary value packs to it).
 */
int ninfer_ternary_unpack(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                          uint64_t payload_bytes, int8_t *values,
                          uint16_t *scales_f16);

/*
 * ninfer_blocks_to_planes / ninfer_planes_to_blocks -- [FMT] §3-§4: the ggml
 * stream of single-group blocks (row-major, groups_per_row blocks per row)
 * <-> the row-split payload. Block layouts: PQ2_0 34 bytes [scale 2][base 32];
 * PTQ1_0 28 bytes [base 24][high 2][scale 2]. The two are exact inverses: bytes
 * are moved, never changed. blocks_bytes must be n * groups_per_row * 34 (28).
 * Host, synchronous. Errors: UNKNOWN_FORMAT, SHAPE, INVALID_ARGUMENT, SIZE_MISMATCH.
 */
int ninfer_blocks_to_planes(int fmt, uint64_t n, uint64_t k, const uint8_t *blocks,
                            uint64_t blocks_bytes, uint8_t *payload,
                            uint64_t payload_bytes);
int ninfer_planes_to_blocks(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                            uint64_t payload_bytes, uint8_t *blocks,
                            uint64_t blocks_bytes);

/*
 * ninfer_blocks_to_planes_device / ninfer_planes_to_blocks_device -- the same
 * two conversions ([FMT] §3-§4 block slices) on device buffers, for a model
 * whose block stream is already in device memory.
 *   blocks: device, n * groups_per_row * 34 (PQ2_0) or 28 (PTQ1_0) bytes,
 *     2-byte aligned; payload: device, payload_bytes of the geometry, 256-byte
 *     aligned. Same bytes out as the host functions (to planes: the gaps between
 *     planes are zero).
 *   Asynchronous on `stream`; the caller keeps both buffers alive until it completes.
 * Errors: UNKNOWN_FORMAT, SHAPE, INVALID_ARGUMENT, SIZE_MISMATCH, ALIGNMENT,
 *   OVERFLOW, CUDA (launch failures), all before any device work is queued
 *   except CUDA.
 */
int ninfer_blocks_to_planes_device(int fmt, uint64_t n, uint64_t k, const uint8_t *blocks,
                                   uint64_t blocks_bytes, uint8_t *payload,
                                   uint64_t payload_bytes, ninfer_stream stream);
int ninfer_planes_to_blocks_device(int fmt, uint64_t n, uint64_t k, const uint8_t *payload,
                                   uint64_t payload_bytes, uint8_t *blocks,
                                   uint64_t blocks_bytes, ninfer_stream stream);

/*
 * ninfer_hadamard_fwd -- [V3] §8 hadamard_signs, [TS] §4.2 forward transform:
 *   for every row m and 1024-block b: y_b = H (D_b * x_b) / sqrt(1024), with H
 *   the unnormalised Sylvester Hadamard matrix in natural order
 *   (H[i][j] = (-1)^popcount(i & j)) and D_b the block's slice of the sign vector.
 * ninfer_hadamard_inv -- [TS] §4.2 inverse (embedding rows): y_b = D_b * (H x_b) / 32.
 *   x: device, M x K row-major of x_dtype; y: device, M x K of y_dtype
 *     (may alias x exactly for in-place use when the dtypes match).
 *   signs_bf16: device bfloat16[K], each +1 or -1 (other values give
 *     unspecified results; they are not checked on the device).
 *   K must be a multiple of 1024 ([V3] §8: "K ... is a multiple of 1024").
 *   Computed in fp32; y rounded to y_dtype.
 * Errors: INVALID_ARGUMENT, SHAPE (K % 1024 != 0), ALIGNMENT, CUDA.
 */
/*
 * ninfer_validate_signs -- load-time check of a hadamard_signs vector ([V3] §8:
 *   bfloat16 [K], K a multiple of 1024, every entry +1 or -1). The device
 *   entry points do not check sign values; validate a vector once with this
 *   when it is loaded.
 *   signs_bf16: host bfloat16[K] (bit patterns 0x3F80 = +1, 0xBF80 = -1).
 * Errors: INVALID_ARGUMENT (NULL, or an entry other than +-1, named in the
 *   message), SHAPE (K == 0 or K % 1024 != 0).
 */
int ninfer_validate_signs(const uint16_t *signs_bf16, uint64_t K);

int ninfer_hadamard_fwd(const void *x, int x_dtype, void *y, int y_dtype,
                        const uint16_t *signs_bf16, uint64_t M, uint64_t K,
                        ninfer_stream stream);
int ninfer_hadamard_inv(const void *x, int x_dtype, void *y, int y_dtype,
                        const uint16_t *signs_bf16, uint64_t M, uint64_t K,
                        ninfer_stream stream);

/*
 * ninfer_ternary_matmul_workspace -- bytes of device workspace that
 * ninfer_ternary_matmul needs for this problem (0 when none). Host only.
 */
int ninfer_ternary_matmul_workspace(int fmt, uint64_t n, uint64_t k, uint64_t M,
                                    int rotate, uint64_t *bytes);

/*
 * ninfer_ternary_matmul -- the rotated ternary projection:
 *   y[m][r] = sum_c W[r][c] * xr[m][c],   W[r][c] = value(code[r][c]) * scale[r][c/128],
 *   xr = forward transform of x (as ninfer_hadamard_fwd) when signs_bf16 != NULL,
 *   xr = x when signs_bf16 == NULL (unrotated use).
 * ([V3] §8: the matrix multiplies hadamard_transform(input, signs) instead of
 * the raw input; [TS] §4.4: forward transform before every low-bit projection
 * and before the output head; value mapping as ninfer_ternary_pack.)
 *   payload: device, the row-split payload of an n x k matrix, exactly
 *     payload_bytes == geometry.payload_bytes, 256-byte aligned.
 *   x: device M x k row-major of x_dtype (f32, bf16 or f16), 16-byte aligned,
 *     row stride k elements.
 *   signs_bf16: device bfloat16[k] (+-1) or NULL; non-NULL requires k % 1024 == 0.
 *   y: device M x n row-major of y_dtype (f32 or bf16).
 *   workspace: device scratch of at least ninfer_ternary_matmul_workspace()
 *     bytes (NULL allowed when that is 0); its contents are not preserved.
 *   M >= 1. Decode shapes (M <= 8) run the fused rotate + decode + GEMV
 *   kernels; larger M run the prefill path.
 * Arithmetic: transform in fp32. M = 1 (both formats): the rotated
 * activations are rounded to 16-bit fixed point per 1024-block (|x16| < 2^14,
 * relative error <= 2^-14 of the block maximum); code x activation products
 * accumulate exactly in int32 per 128-weight group, then scale in fp32
 * (PTQ1_0 shapes the M = 1 kernel cannot split among at most four CTAs of a
 * cluster -- more than 2048 groups per row, or more than 512 with over about
 * 147,000 rows -- take the 2 <= M <= 8 path below).
 * 2 <= M <= 8 (both formats): binary16 activations scaled per 1024-block
 * (relative error <= 2^-11 per element), exact binary16 codes, products on the
 * tensor cores (mma.sync) with fp32 accumulation. M > 8 (prefill, both
 * formats): binary16 activations and the exact binary16 weights
 * (code - 1) * scale on the tensor cores (tcgen05), fp32 accumulation; PTQ1_0
 * planes are first rewritten exactly as PQ2_0 planes in the workspace. Inputs
 * no fast path takes (raw x whose rows are not 16-byte aligned, M > 8 with
 * k % 1024 != 0) run a general tiled kernel in fp32. The infinity-norm relative
 * error against the exact result stays under 1e-3 on the decode paths and
 * under 2e-2 on the prefill path.
 * Errors: INVALID_ARGUMENT, UNKNOWN_FORMAT, SHAPE, SIZE_MISMATCH, ALIGNMENT, CUDA.
 */
int ninfer_ternary_matmul(int fmt, const uint8_t *payload, uint64_t payload_bytes,
                          uint64_t n, uint64_t k, const void *x, int x_dtype,
                          const uint16_t *signs_bf16, void *y, int y_dtype,
                          uint64_t M, void *workspace, uint64_t workspace_bytes,
                          ninfer_stream stream);

/*
 * ninfer_ternary_gate_up -- the FFN gate and up projections of one activation
 * with the SwiGLU product ([TS] §4.2: fused gate/up weights keep each original
 * projection's transform; §4.4: the dense gated FFN, read as SwiGLU):
 *   y[m][r] = silu(g[m][r]) * u[m][r],  silu(a) = a / (1 + e^-a),
 *   g = ninfer_ternary_matmul(payload_gate, x, signs_gate),
 *   u = ninfer_ternary_matmul(payload_up, x, signs_up).
 *   payload_gate, payload_up: device, the same format and shape n x k
 *     (payload_bytes each, 256-byte aligned).
 *   signs_gate_bf16, signs_up_bf16: both device bfloat16[k], or both NULL (no
 *     rotation); they may be the same pointer (one rotation serves both).
 *   x, y, x_dtype, y_dtype, M, stream: as ninfer_ternary_matmul.
 *   workspace: device scratch of at least ninfer_ternary_gate_up_workspace()
 *     bytes, 256-byte aligned (NULL allowed when that is 0). PQ2_0 with M = 1
 *     runs both projections and the product in one kernel and needs none;
 *     other cases keep fp32 g and u in the workspace.
 * Errors: as ninfer_ternary_matmul; INVALID_ARGUMENT when exactly one sign
 *   vector is given.
 * ninfer_ternary_gate_up_workspace: the workspace bytes of a call with these
 *   fmt, n, k, M, with rotate != 0 when sign vectors are given and
 *   distinct_signs != 0 when they are two different pointers (0 when the
 *   single-kernel path applies). Errors: as ninfer_ternary_geometry, SHAPE for M = 0.
 */
int ninfer_ternary_gate_up_workspace(int fmt, uint64_t n, uint64_t k, uint64_t M,
                                     int rotate, int distinct_signs, uint64_t *bytes);
int ninfer_ternary_gate_up(int fmt, const uint8_t *payload_gate, const uint8_t *payload_up,
                           uint64_t payload_bytes, uint64_t n, uint64_t k,
                           const void *x, int x_dtype, const uint16_t *signs_gate_bf16,
                           const uint16_t *signs_up_bf16, void *y, int y_dtype, uint64_t M,
                           void *workspace, uint64_t workspace_bytes, ninfer_stream stream);

/*
 * ninfer_ternary_embed -- embedding rows ([TS] §4.4: token id -> low-bit
 * embedding row -> inverse signed Hadamard transform; [V3] §7.3: a row range of
 * a row-split matrix spans intervals of the base, high and scale planes):
 *   out[i][c] = inverse transform of (W[ids[i]][:]) , i < count.
 *   payload: device row-split payload of the n x k embedding matrix.
 *   ids: device int32[count]; an id outside [0, n) writes a zero row and sets
 *     bit 0 of *status_dev (if status_dev != NULL; never cleared by the library).
 *   signs_bf16: device bfloat16[k] (+-1), k % 1024 == 0; NULL skips the transform.
 *   out: device count x k of out_dtype (f32 or bf16).
 * Errors: INVALID_ARGUMENT, UNKNOWN_FORMAT, SHAPE, SIZE_MISMATCH, ALIGNMENT, CUDA.
 */
int ninfer_ternary_embed(int fmt, const uint8_t *payload, uint64_t payload_bytes,
                         uint64_t n, uint64_t k, const int32_t *ids, uint64_t count,
                         const uint16_t *signs_bf16, void *out, int out_dtype,
                         int32_t *status_dev, ninfer_stream stream);

/*
 * ninfer_device_errors -- reads the library's device error word on the current
 * device into *out and clears it when clear != 0. Bit 0 (value 1): a kernel
 * gave up waiting for its own asynchronous weight copies (a bounded wait of
 * about two seconds ran out); that call's output is incomplete. Kernels never
 * trap; this word is how such a failure is reported. Host, synchronous.
 * Errors: INVALID_ARGUMENT (out NULL), CUDA.
 */
int ninfer_device_errors(uint32_t *out, int clear);

/*
 * ninfer_set_wait_limit -- bound, in SM clock cycles, of each wait of the
 * M = 1 decode kernels of both formats (ninfer_ternary_matmul and the
 * one-kernel ninfer_ternary_gate_up) for their weight copies, for calls launched after
 * this one; the default is 4e9 (about two seconds). No counterpart on the
 * source pages: a diagnostic hook that lets a test drive the failure path
 * described under ninfer_device_errors without breaking anything. cycles == 0
 * makes every such wait give up at its first check even when the copy has
 * landed: the call then returns NINFER_OK, sets bit 0 of the error word,
 * leaves its output incomplete, and its CTAs let the copies already issued
 * land before they exit. Other kernels keep their fixed bound. Process-wide,
 * host only. Errors: INVALID_ARGUMENT (cycles < 0).
 */
int ninfer_set_wait_limit(long long cycles);

/*
 * ninfer_set_prefetch_before_dependency -- process-wide switch, default 1.
 * With 1, decode projections (ninfer_ternary_matmul with M <= 8) are launched
 * with programmatic dependent launch: they begin streaming the weight payload
 * while the preceding work on the stream is still finishing, and touch the
 * activations, signs and output only after it has completed. Set 0 when the
 * work immediately preceding a call writes that call's weight payload.
 * Always returns NINFER_OK.
 */
int ninfer_set_prefetch_before_dependency(int enable);

/*
 * ninfer_ternary_matmul_noalloc -- ninfer_ternary_matmul for callers that
 * cannot allocate device memory. No counterpart on the source pages: it is a
 * convenience of this library.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator around the
 * projection -- for instance a plug-in whose host hands it only the input and
 * output buffers, or a runtime with no device allocator of its own. Such a
 * caller cannot provide the workspace ninfer_ternary_matmul asks for on the
 * paths that stage rotated activations.
 *
 * What it does: exactly ninfer_ternary_matmul (same arguments minus the
 * workspace, same results), with the workspace taken from a fixed array of
 * NINFER_NOALLOC_SCRATCH_BYTES bytes that the library keeps in device memory.
 * Every GPU that loads the library holds that array until the process exits.
 * The call itself allocates nothing.
 *   - Limit: a problem whose ninfer_ternary_matmul_workspace() exceeds
 *     NINFER_NOALLOC_SCRATCH_BYTES is rejected with NINFER_ERR_SIZE_MISMATCH
 *     (use ninfer_ternary_matmul with your own workspace instead).
 *   - Set-up: the first call on a device (with that device current) looks up
 *     the array's device address once; make that first call before any stream
 *     capture. The address is kept for the life of the process, so calls must
 *     not cross a cudaDeviceReset or any other teardown of the device's
 *     primary context.
 *   - Sharing: all calls on a device share the one array and it keeps the last
 *     call's contents (every call overwrites what it reads, so no clearing is
 *     needed). Calls that may overlap on the GPU -- on different streams, or
 *     from different host threads without ordering -- race on the array; order
 *     them on one stream.
 * Errors: as ninfer_ternary_matmul, plus SIZE_MISMATCH for the limit above.
 */
#define NINFER_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
int ninfer_ternary_matmul_noalloc(int fmt, const uint8_t *payload, uint64_t payload_bytes,
                                  uint64_t n, uint64_t k, const void *x, int x_dtype,
                                  const uint16_t *signs_bf16, void *y, int y_dtype,
                                  uint64_t M, ninfer_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* NINFER_TERNARY_H */
