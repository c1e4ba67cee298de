"""fp64 CPU oracle: row-split ternary planes, block Hadamard transform, projection.

TEST INFRASTRUCTURE ONLY. Imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg; never by the product library.

Each function restates one step of the source pages in plain numpy (float64,
or exact integers for the codec), with no blocking, fusion or reordering
beyond what the step's own definition states:

* geometry          -- "bonsai三元GGUF模型转ninfer模型01" §3 (row-split plane geometry)
* codec             -- same page §2/§3 (per-group base/high/scale bytes),
                       "GGUF 完整讲解" §4.3 (Q2_0 2-bit field order and the
                       offset mapping code -> code - 1),
                       the base-3 reading for PTQ1_0 (the pages give 24 + 2
                       bytes for 128 three-valued weights but no digit order)
* block <-> plane   -- "bonsai三元GGUF模型转ninfer模型01" §3 (block byte order)
                       and §4 (BLOCK_PLANE_SLICES)
* transform         -- "artifact-container.md" §8 (hadamard_signs: sign multiply
                       per 1024-block, then the normalised Sylvester
                       Walsh-Hadamard transform) and the TensorSharp article §4.2
                       (forward H(D.x)/sqrt(1024), inverse D.(H.x)/sqrt(1024))
* projection        -- y = W . transform(x) with W[r, c] = value(code) * scale
                       of the group (format page §3: one binary16 per group)
* embedding         -- inverse transform of gathered rows (TensorSharp article §4.4)
* error figures     -- the infinity-norm relative error the accuracy bounds are
                       stated in, and a per-element relative error over the
                       outputs that are not small (the pages fix no metric)

Parity pins: all functions are pinned in tests/test_oracle_pins.py.
"""
from __future__ import annotations

from collections import namedtuple

import numpy as np

GROUP = 128              # weights per group, both ternary formats
PLANE_ALIGNMENT = 256    # plane start alignment (format page §1 constants)
HADAMARD_BLOCK = 1024    # transform block size (format page §6 constants)

# (name, group_size, base_bytes, high_bytes) -- format page §2.
TernaryFormat = namedtuple("TernaryFormat", "name group base_bytes high_bytes")
FORMATS = {
    "PQ2_0_G128": TernaryFormat("PQ2_0_G128", 128, 32, 0),
    "PTQ1_0_G128": TernaryFormat("PTQ1_0_G128", 128, 24, 2),
}

# Field order of RowSplitGeometry -- format page §3.
GEOMETRY_FIELDS = (
    "n", "k", "k_pad", "groups_per_row", "base_bytes_per_group",
    "high_bytes_per_group", "base_row_bytes", "high_row_bytes",
    "scale_row_bytes", "base_offset", "base_bytes", "high_offset",
    "high_bytes", "scale_offset", "scale_bytes", "payload_bytes",
)
RowSplitGeometry = namedtuple("RowSplitGeometry", GEOMETRY_FIELDS)

# ggml single-group block layouts -- format page §3 ("plane order != in-block
# byte order") and §4: (start, stop) byte ranges for (base, high, scale).
GGML_BLOCK_BYTES = {"PQ2_0_G128": 34, "PTQ1_0_G128": 28}
BLOCK_PLANE_SLICES = {
    "PQ2_0_G128": ((2, 34), None, (0, 2)),          # [scale 2][qs 32]
    "PTQ1_0_G128": ((0, 24), (24, 26), (26, 28)),   # [qs 24][qh 2][scale 2]
}


def _align_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


def _fmt(fmt) -> TernaryFormat:
    if isinstance(fmt, TernaryFormat):
        return fmt
    if fmt not in FORMATS:
        raise ValueError(f"unknown numeric format: {fmt!r}")
    return FORMATS[fmt]


# ----------------------------------------------------------------------------
# geometry (format page §3)
# ----------------------------------------------------------------------------
def row_split_geometry(fmt, n: int, k: int) -> RowSplitGeometry:
    """The 16 RowSplitGeometry fields for an n x k matrix, in the page's order.

    k_pad = align_up(k, 128); groups = k_pad / 128; per-row bytes are groups
    times the per-group byte counts (2 scale bytes per group); the base plane
    starts at 0, the high plane at align_up(base_bytes, 256) (even when empty)
    and the scale plane 256-aligned after it. The plane sizes are n times the
    per-row sizes.
    """
    f = _fmt(fmt)
    n, k = int(n), int(k)
    if n <= 0 or k <= 0:
        raise ValueError("shape must be rank 2 with positive dimensions")
    k_pad = _align_up(k, f.group)
    groups = k_pad // f.group
    base_row = groups * f.base_bytes
    high_row = groups * f.high_bytes
    scale_row = groups * 2
    base_offset = 0
    base_bytes = n * base_row
    high_offset = _align_up(base_offset + base_bytes, PLANE_ALIGNMENT)
    high_bytes = n * high_row
    scale_offset = high_offset + _align_up(high_bytes, PLANE_ALIGNMENT)
    scale_bytes = n * scale_row
    payload = scale_offset + scale_bytes
    return RowSplitGeometry(n, k, k_pad, groups, f.base_bytes, f.high_bytes,
                            base_row, high_row, scale_row, base_offset,
                            base_bytes, high_offset, high_bytes, scale_offset,
                            scale_bytes, payload)


# ----------------------------------------------------------------------------
# per-group codec
# ----------------------------------------------------------------------------
# PQ2_0: 32 base bytes hold the group's 128 weights in order, four per byte,
# weight j in bits 2*(j % 4) of byte j // 4 (least significant field first);
# the field is an offset code: value = code - 1 (00 -> -1, 01 -> 0, 10 -> +1,
# 11 -> +2, as in the Q2_0 dequantisation routine of "GGUF 完整讲解" §4.3).
#
# PTQ1_0: 24 base bytes + 2 high bytes hold 128 three-valued weights. Reading:
# t = value + 1 in {0, 1, 2}; base byte b holds weights 5b .. 5b+4 as
# sum_i t[5b+i] * 3**i; high byte h holds weights 120+4h .. 120+4h+3 as
# sum_i t[120+4h+i] * 3**i (little-endian base-3 digits, weights in order).

def _group_codes_pq2(values_g: np.ndarray) -> np.ndarray:
    """(..., 128) values -> (..., 32) base bytes."""
    c = (values_g.astype(np.int64) + 1).reshape(values_g.shape[:-1] + (32, 4))
    byte = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    return byte.astype(np.uint8)


def _group_codes_ptq1(values_g: np.ndarray):
    """(..., 128) values -> ((..., 24) base bytes, (..., 2) high bytes)."""
    t = values_g.astype(np.int64) + 1
    lead = values_g.shape[:-1]
    qs = t[..., :120].reshape(lead + (24, 5))
    qh = t[..., 120:].reshape(lead + (2, 4))
    base = sum(qs[..., i] * 3 ** i for i in range(5))
    high = sum(qh[..., i] * 3 ** i for i in range(4))
    return base.astype(np.uint8), high.astype(np.uint8)


def _decode_pq2(base_g: np.ndarray) -> np.ndarray:
    """(..., 32) base bytes -> (..., 128) values (code - 1); code 3 reads +2."""
    b = base_g.astype(np.int64)
    fields = [((b >> (2 * i)) & 3) for i in range(4)]          # weight 4j + i
    codes = np.stack(fields, axis=-1).reshape(base_g.shape[:-1] + (128,))
    return codes - 1


def _decode_ptq1(base_g: np.ndarray, high_g: np.ndarray) -> np.ndarray:
    """(..., 24) base + (..., 2) high bytes -> (..., 128) values (digit - 1).

    Digits are taken as (byte // 3**i) % 3, which is the inverse of the
    packing above for every valid byte (< 243 base, < 81 high) and is the
    defined reading of the remaining byte values.
    """
    b = base_g.astype(np.int64)
    h = high_g.astype(np.int64)
    lead = base_g.shape[:-1]
    lo = np.stack([(b // 3 ** i) % 3 for i in range(5)], axis=-1).reshape(lead + (120,))
    hi = np.stack([(h // 3 ** i) % 3 for i in range(4)], axis=-1).reshape(lead + (8,))
    return np.concatenate([lo, hi], axis=-1) - 1


def _check_values(values: np.ndarray):
    if values.ndim != 2:
        raise ValueError("values must be n x k")
    if values.size and (values.min() < -1 or values.max() > 1):
        raise ValueError("ternary values must be -1, 0 or +1")


def pack_planes(fmt, values: np.ndarray, scales_f16: np.ndarray) -> np.ndarray:
    """values (n x k, in {-1,0,1}) + binary16 scales (n x groups) -> payload bytes.

    Pad weights (columns k .. k_pad-1) encode value 0. Planes are row-major
    [row][group][bytes]; the scale plane stores binary16 little-endian.
    """
    f = _fmt(fmt)
    values = np.asarray(values)
    _check_values(values)
    n, k = values.shape
    g = row_split_geometry(f, n, k)
    scales_f16 = np.asarray(scales_f16, dtype=np.uint16)
    if scales_f16.shape != (n, g.groups_per_row):
        raise ValueError("scales must be n x groups_per_row binary16 words")
    padded = np.zeros((n, g.k_pad), dtype=np.int64)
    padded[:, :k] = values
    grouped = padded.reshape(n, g.groups_per_row, GROUP)
    payload = np.zeros(g.payload_bytes, dtype=np.uint8)
    if f.name == "PQ2_0_G128":
        base = _group_codes_pq2(grouped)
        payload[g.base_offset:g.base_offset + g.base_bytes] = base.reshape(-1)
    else:
        base, high = _group_codes_ptq1(grouped)
        payload[g.base_offset:g.base_offset + g.base_bytes] = base.reshape(-1)
        payload[g.high_offset:g.high_offset + g.high_bytes] = high.reshape(-1)
    payload[g.scale_offset:g.scale_offset + g.scale_bytes] = (
        scales_f16.astype("<u2").reshape(-1).view(np.uint8))
    return payload


def _planes(f: TernaryFormat, g: RowSplitGeometry, payload: np.ndarray):
    payload = np.asarray(payload, dtype=np.uint8).reshape(-1)
    if payload.size != g.payload_bytes:
        raise ValueError(f"payload stores {payload.size} bytes; layout requires {g.payload_bytes}")
    base = payload[g.base_offset:g.base_offset + g.base_bytes].reshape(
        g.n, g.groups_per_row, f.base_bytes)
    high = None
    if f.high_bytes:
        high = payload[g.high_offset:g.high_offset + g.high_bytes].reshape(
            g.n, g.groups_per_row, f.high_bytes)
    scales = payload[g.scale_offset:g.scale_offset + g.scale_bytes].view("<u2").reshape(
        g.n, g.groups_per_row)
    return base, high, scales


def unpack_planes(fmt, n: int, k: int, payload: np.ndarray):
    """Inverse of pack_planes: -> (values n x k int8, scales n x groups uint16).

    Raises ValueError on a code that no ternary value packs to (PQ2_0 code 3,
    PTQ1_0 base byte >= 243 or high byte >= 81).
    """
    f = _fmt(fmt)
    g = row_split_geometry(f, n, k)
    base, high, scales = _planes(f, g, payload)
    if f.name == "PQ2_0_G128":
        vals = _decode_pq2(base)
        if (vals > 1).any():
            raise ValueError("invalid PQ2_0 code 3")
    else:
        if (base >= 243).any() or (high >= 81).any():
            raise ValueError("invalid PTQ1_0 base-3 byte")
        vals = _decode_ptq1(base, high)
    vals = vals.reshape(g.n, g.k_pad)[:, :g.k].astype(np.int8)
    return vals, np.array(scales, dtype=np.uint16)


def dequantize(fmt, payload: np.ndarray, n: int, k: int, rows=None) -> np.ndarray:
    """Dense fp64 weights W[r, c] = value(code[r, c]) * scale[r, c // 128], c < k.

    rows selects a subset of output rows (all rows when None). Each row's group
    g is read from base_offset + r*base_row_bytes + g*base_bytes_per_group (and
    likewise for the high plane) and scale_offset + r*scale_row_bytes + 2g.
    """
    f = _fmt(fmt)
    g = row_split_geometry(f, n, k)
    base, high, scales = _planes(f, g, payload)
    rows = np.arange(g.n) if rows is None else np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= g.n):
        raise ValueError("row index out of range")
    if f.name == "PQ2_0_G128":
        vals = _decode_pq2(base[rows])
    else:
        vals = _decode_ptq1(base[rows], high[rows])
    s = np.ascontiguousarray(scales[rows]).view("<f2").astype(np.float64)   # exact widening
    w = vals.astype(np.float64) * s[:, :, None]
    return w.reshape(rows.size, g.k_pad)[:, :g.k]


# ----------------------------------------------------------------------------
# ggml block stream <-> planes (format page §3, §4)
# ----------------------------------------------------------------------------
def planes_to_blocks(fmt, n: int, k: int, payload: np.ndarray) -> np.ndarray:
    """Row-split payload -> the ggml stream of single-group blocks, row-major."""
    f = _fmt(fmt)
    g = row_split_geometry(f, n, k)
    base, high, scales = _planes(f, g, payload)
    nb = GGML_BLOCK_BYTES[f.name]
    sb, sh, ss = BLOCK_PLANE_SLICES[f.name]
    blocks = np.zeros((g.n, g.groups_per_row, nb), dtype=np.uint8)
    blocks[:, :, sb[0]:sb[1]] = base
    if sh is not None:
        blocks[:, :, sh[0]:sh[1]] = high
    blocks[:, :, ss[0]:ss[1]] = scales.astype("<u2").view(np.uint8).reshape(g.n, g.groups_per_row, 2)
    return blocks.reshape(-1)


def blocks_to_planes(fmt, n: int, k: int, blocks: np.ndarray) -> np.ndarray:
    """Inverse of planes_to_blocks (exact: every byte moves, none is changed)."""
    f = _fmt(fmt)
    g = row_split_geometry(f, n, k)
    nb = GGML_BLOCK_BYTES[f.name]
    blocks = np.asarray(blocks, dtype=np.uint8).reshape(-1)
    if blocks.size != g.n * g.groups_per_row * nb:
        raise ValueError("block stream size does not match the shape")
    blocks = blocks.reshape(g.n, g.groups_per_row, nb)
    sb, sh, ss = BLOCK_PLANE_SLICES[f.name]
    payload = np.zeros(g.payload_bytes, dtype=np.uint8)
    payload[g.base_offset:g.base_offset + g.base_bytes] = blocks[:, :, sb[0]:sb[1]].reshape(-1)
    if sh is not None:
        payload[g.high_offset:g.high_offset + g.high_bytes] = blocks[:, :, sh[0]:sh[1]].reshape(-1)
    payload[g.scale_offset:g.scale_offset + g.scale_bytes] = blocks[:, :, ss[0]:ss[1]].reshape(-1)
    return payload


# ----------------------------------------------------------------------------
# block Hadamard transform ("artifact-container.md" §8; TensorSharp §4.2)
# ----------------------------------------------------------------------------
_H_CACHE = {}


def hadamard_matrix(size: int = HADAMARD_BLOCK) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix, natural order:
    H[i, j] = (-1) ** popcount(i & j)."""
    if size in _H_CACHE:
        return _H_CACHE[size]
    if size <= 0 or size & (size - 1):
        raise ValueError("size must be a power of two")
    idx = np.arange(size, dtype=np.int64)
    ij = np.bitwise_and.outer(idx, idx)
    parity = np.zeros_like(ij)
    for bit in range(int(size).bit_length()):
        parity ^= (ij >> bit) & 1
    H = (1 - 2 * parity).astype(np.float64)
    _H_CACHE[size] = H
    return H


def _check_signs(signs, K: int) -> np.ndarray:
    D = np.asarray(signs, dtype=np.float64).reshape(-1)
    if D.size != K:
        raise ValueError("sign vector length must equal the input width")
    if not np.all(np.abs(D) == 1.0):
        raise ValueError("sign vector elements must be +1 or -1")
    return D


def _blocks(x, signs):
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    K = x.shape[1]
    if K % HADAMARD_BLOCK:
        raise ValueError("width must be a multiple of the 1024-element block")
    return x, _check_signs(signs, K), K // HADAMARD_BLOCK


def hadamard_forward(x, signs) -> np.ndarray:
    """Per 1024-block b of every row: xr_b = H (D_b * x_b) / sqrt(1024)."""
    x, D, nblk = _blocks(x, signs)
    H = hadamard_matrix()
    out = np.empty_like(x)
    for b in range(nblk):
        s = slice(b * HADAMARD_BLOCK, (b + 1) * HADAMARD_BLOCK)
        out[:, s] = (H @ (D[s] * x[:, s]).T).T / 32.0
    return out


def hadamard_inverse(x, signs) -> np.ndarray:
    """Per 1024-block b of every row: out_b = D_b * (H x_b) / sqrt(1024)."""
    x, D, nblk = _blocks(x, signs)
    H = hadamard_matrix()
    out = np.empty_like(x)
    for b in range(nblk):
        s = slice(b * HADAMARD_BLOCK, (b + 1) * HADAMARD_BLOCK)
        out[:, s] = D[s] * (H @ x[:, s].T).T / 32.0
    return out


# ----------------------------------------------------------------------------
# projection and embedding
# ----------------------------------------------------------------------------
def ternary_matmul(fmt, payload, n: int, k: int, x, signs=None, rows=None) -> np.ndarray:
    """y[m, r] = sum_c W[r, c] * xr[m, c], xr = forward transform of x
    (x itself when signs is None). Returns M x len(rows) in fp64."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    if x.shape[1] != k:
        raise ValueError("activation width must equal k")
    xr = x if signs is None else hadamard_forward(x, signs)
    W = dequantize(fmt, payload, n, k, rows)
    return xr @ W.T


def gate_up_swiglu(fmt, payload_gate, payload_up, n: int, k: int, x, signs_gate=None, signs_up=None,
                   rows=None) -> np.ndarray:
    """FFN gate/up with the SwiGLU product, fp64: y = silu(g) * u with
    g = ternary_matmul(gate, x, signs_gate), u = ternary_matmul(up, x, signs_up)
    and silu(a) = a / (1 + e^-a). Fused gate/up weights keep each original
    projection's transform (TensorSharp article section 4.2); the layers' dense
    gated FFN (section 4.4) is read as SwiGLU."""
    g = ternary_matmul(fmt, payload_gate, n, k, x, signs_gate, rows)
    u = ternary_matmul(fmt, payload_up, n, k, x, signs_up, rows)
    return g / (1.0 + np.exp(-g)) * u


def embed_rows(fmt, payload, n: int, k: int, ids, signs) -> np.ndarray:
    """out_i = inverse transform of dequantised row ids[i] (count x k, fp64)."""
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= n):
        raise ValueError("token id out of range")
    W = dequantize(fmt, payload, n, k, ids)
    return hadamard_inverse(W, signs)


def max_rel_error(got, ref) -> float:
    """Infinity-norm relative error, max_i |got_i - ref_i| / max_i |ref_i|: the
    accuracy figure the decode, transform and embedding bounds (1e-3) and the
    tensor-core prefill bound (2e-2) are stated in. The pages fix no metric; this
    is the plain reading of "max relative error" for a vector result. The
    denominator is always the reference's. With an all-zero (or empty)
    reference the relative error is undefined and the absolute error
    max_i |got_i - ref_i| is returned instead, so an exact zero output scores 0."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    return float(num / den) if den > 0 else float(num)


def significant_rel_error(got, ref, floor: float = 0.1) -> float:
    """Per-element relative error over the outputs that are not small:
    max_i |got_i - ref_i| / |ref_i| over the i with |ref_i| >= floor * rms(ref),
    rms(ref) = sqrt(mean(ref_i^2)). It catches a localised error on small
    outputs (a wrong row or group with a small value) that the infinity-norm
    figure hides under a large max |ref|. 0.0 when no element qualifies (an
    empty or all-zero reference)."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    if got.shape != ref.shape:
        raise ValueError("got and ref differ in size")
    if ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref))
    sel = (np.abs(ref) >= floor * rms) & (ref != 0)
    if not np.any(sel):
        return 0.0
    return float(np.max(np.abs(got[sel] - ref[sel]) / np.abs(ref[sel])))
