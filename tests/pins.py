"""Pins for the CPU oracle: each function checks the oracle against something
other than itself (values printed on the pages, a library routine, a closed
form, an invariant, or brute force on tiny inputs).

The functions raise AssertionError on failure. test_oracle_pins.py runs them
as tests; test_oracle_mutations.py plants mistakes in the oracle and checks
that at least one pin catches each mistake.
"""
import numpy as np
import scipy.linalg

import oracle
import synth
from conftest import read_golden

ORDER = oracle.GEOMETRY_FIELDS


def _hex_bytes(tokens):
    return np.array([int(t, 16) for t in tokens], dtype=np.uint8)


# ---------------------------------------------------------------- geometry ---
def pin_geometry_printed():
    """Printed sizes/offsets (format page §3) reproduce exactly."""
    for fmt, n, k, field, value in read_golden("geometry_pins.txt"):
        g = oracle.row_split_geometry(fmt, int(n), int(k))
        assert getattr(g, field) == int(value), (fmt, n, k, field, getattr(g, field), value)


def pin_geometry_scale_start_table():
    """Scale plane starts at rows*groups*32 (PQ2_0) / rows*groups*26 (PTQ1_0)
    wherever the plane sizes are 256-multiples (every workload shape), and
    PQ2_0's empty high plane sits at the scale offset."""
    for n, k in [(256, 1024), (17408, 5120), (5120, 17408), (248320, 5120), (2048, 6144)]:
        p = oracle.row_split_geometry("PQ2_0_G128", n, k)
        t = oracle.row_split_geometry("PTQ1_0_G128", n, k)
        assert p.scale_offset == n * p.groups_per_row * 32
        assert t.scale_offset == n * t.groups_per_row * 26
        assert p.high_offset == p.scale_offset and p.high_bytes == 0
        # 34 / 28 bytes per group in total (2.125 / 1.75 bits per weight)
        assert p.payload_bytes == n * p.groups_per_row * 34
        assert t.payload_bytes == n * t.groups_per_row * 28


def pin_geometry_field_order_and_alignment():
    """Field order as printed; planes 256-aligned and disjoint; k_pad = align_up(k,128)."""
    assert tuple(oracle.GEOMETRY_FIELDS) == (
        "n", "k", "k_pad", "groups_per_row", "base_bytes_per_group",
        "high_bytes_per_group", "base_row_bytes", "high_row_bytes",
        "scale_row_bytes", "base_offset", "base_bytes", "high_offset",
        "high_bytes", "scale_offset", "scale_bytes", "payload_bytes")
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 5000))
        k = int(rng.integers(1, 20000))
        for fmt, (b, h) in {"PQ2_0_G128": (32, 0), "PTQ1_0_G128": (24, 2)}.items():
            g = oracle.row_split_geometry(fmt, n, k)
            assert g.k_pad % 128 == 0 and g.k <= g.k_pad < g.k + 128
            assert (g.base_bytes_per_group, g.high_bytes_per_group) == (b, h)
            assert g.base_offset == 0 and g.high_offset % 256 == 0 and g.scale_offset % 256 == 0
            assert g.high_offset >= g.base_bytes and g.scale_offset >= g.high_offset + g.high_bytes
            assert g.high_offset - g.base_bytes < 256
            assert g.scale_offset - (g.high_offset + g.high_bytes) < 256
            assert g.payload_bytes == g.scale_offset + n * g.groups_per_row * 2


# ------------------------------------------------------------------- codec ---
def pin_q2_0_fields():
    """Hand-worked 2-bit fields of the Q2_0 routine (GGUF explainer §4.3)."""
    rows = read_golden("q2_0_fields.txt")
    for r in rows:
        byte = int(r[0], 16)
        want = [int(v) for v in r[1:]]
        # one group whose byte 0 is the fixture byte and the rest code 01 (value 0)
        payload = np.zeros(oracle.row_split_geometry("PQ2_0_G128", 1, 128).payload_bytes, np.uint8)
        payload[:32] = 0x55
        payload[0] = byte
        payload[32 if False else 256:258] = np.array([0x00, 0x3C], np.uint8)   # scale 1.0
        w = oracle.dequantize("PQ2_0_G128", payload, 1, 128)
        assert list(w[0, :4]) == want, (hex(byte), list(w[0, :4]), want)
        assert np.all(w[0, 4:] == 0)


def pin_ptq1_0_digits():
    """Hand-worked base-3 examples of the PTQ1_0 reading."""
    for plane, byte, *vals in read_golden("ptq1_0_digits.txt"):
        g = oracle.row_split_geometry("PTQ1_0_G128", 1, 128)
        payload = np.zeros(g.payload_bytes, np.uint8)
        payload[g.base_offset:g.base_offset + 24] = 121      # all-zero weights
        payload[g.high_offset:g.high_offset + 2] = 40
        payload[g.scale_offset:g.scale_offset + 2] = [0x00, 0x3C]
        if plane == "base":
            payload[g.base_offset + 3] = int(byte)           # weights 15..19
            got = oracle.dequantize("PTQ1_0_G128", payload, 1, 128)[0, 15:20]
        else:
            payload[g.high_offset + 1] = int(byte)           # weights 124..127
            got = oracle.dequantize("PTQ1_0_G128", payload, 1, 128)[0, 124:128]
        assert list(got) == [int(v) for v in vals], (plane, byte, list(got), vals)


def pin_codec_brute_force():
    """Every code/digit pattern: pack -> unpack is the identity, and the
    decoded weight equals value * scale (brute force over all patterns)."""
    # PQ2_0: all 3^4 value quadruples in every byte position of a group
    quads = np.array(np.meshgrid(*[[-1, 0, 1]] * 4, indexing="ij")).reshape(4, -1).T   # 81 x 4
    vals = np.zeros((81, 128), np.int8)
    for pos in range(32):
        vals[:, 4 * pos:4 * pos + 4] = quads
    # PTQ1_0: all 3^5 quintuples in base byte 0 and all 3^4 quadruples in high byte 1
    quint = np.array(np.meshgrid(*[[-1, 0, 1]] * 5, indexing="ij")).reshape(5, -1).T  # 243 x 5
    tvals = np.zeros((243, 128), np.int8)
    tvals[:, 0:5] = quint
    tvals[:81, 124:128] = quads
    for fmt, v in [("PQ2_0_G128", vals), ("PTQ1_0_G128", tvals)]:
        n = v.shape[0]
        scales = synth.f16_bits(np.linspace(0.005, 0.05, n)).reshape(n, 1)
        payload = oracle.pack_planes(fmt, v, scales)
        v2, s2 = oracle.unpack_planes(fmt, n, 128, payload)
        assert np.array_equal(v2, v) and np.array_equal(s2, scales)
        W = oracle.dequantize(fmt, payload, n, 128)
        assert np.array_equal(W, v * scales.view(np.float16).astype(np.float64))
    # every PTQ1_0 byte value < 243 decodes to digits that re-encode to it
    g = oracle.row_split_geometry("PTQ1_0_G128", 243, 128)
    payload = np.zeros(g.payload_bytes, np.uint8)
    base = np.full((243, 24), 121, np.uint8)
    base[:, 0] = np.arange(243)
    payload[:g.base_bytes] = base.reshape(-1)
    payload[g.high_offset:g.high_offset + g.high_bytes] = 40
    payload[g.scale_offset:] = np.tile(np.array([0, 0x3C], np.uint8), 243)
    v, _ = oracle.unpack_planes("PTQ1_0_G128", 243, 128, payload)
    t = v[:, :5].astype(np.int64) + 1
    assert np.array_equal(sum(t[:, i] * 3 ** i for i in range(5)), np.arange(243))


def pin_scale_offset_invariant():
    """Right scale offset -> every scale finite and in [0.005, 0.05]; reading
    PTQ1_0 scales at rows*groups*base_bytes (inside the high plane, the mistake
    the format page §3 warns about) breaks that invariant."""
    c = synth.make_case("down", n=64, k=17408)
    payload = oracle.pack_planes("PTQ1_0_G128", c.values, c.scales)
    g = oracle.row_split_geometry("PTQ1_0_G128", 64, 17408)
    right = payload[g.scale_offset:g.scale_offset + g.scale_bytes].view("<f2").astype(np.float64)
    assert np.all(np.isfinite(right)) and right.min() >= 0.005 and right.max() <= 0.05
    wrong_at = 64 * g.groups_per_row * 24
    wrong = payload[wrong_at:wrong_at + g.scale_bytes].view("<f2").astype(np.float64)
    ok = np.isfinite(wrong) & (wrong >= 0.005) & (wrong <= 0.05)
    assert ok.mean() < 0.5
    # the oracle's own dequantisation reads only in-range scales
    W = oracle.dequantize("PTQ1_0_G128", payload, 64, 17408)
    mags = np.unique(np.abs(W[W != 0]))
    assert mags.min() >= 0.005 and mags.max() <= 0.05


def pin_block_plane_worked():
    """Hand-built single-group blocks <-> planes (format page §3/§4)."""
    for fmt, name, pay in [("PQ2_0_G128", "blocks_pq2_0.txt", 258),
                           ("PTQ1_0_G128", "blocks_ptq1_0.txt", 514)]:
        rows = read_golden(name)
        block = _hex_bytes(rows[0])
        assert block.size == {"PQ2_0_G128": 34, "PTQ1_0_G128": 28}[fmt]
        g = oracle.row_split_geometry(fmt, 1, 128)
        assert g.payload_bytes == pay
        want = np.zeros(pay, np.uint8)
        for r in rows[1:]:
            off = {"base": g.base_offset, "high": g.high_offset, "scale": g.scale_offset}[r[0]]
            data = _hex_bytes(r[1:])
            want[off:off + data.size] = data
        got = oracle.blocks_to_planes(fmt, 1, 128, block)
        assert np.array_equal(got, want)
        assert np.array_equal(oracle.planes_to_blocks(fmt, 1, 128, got), block)


def pin_block_plane_roundtrip():
    """Slices cover each block exactly; planes->blocks->planes and
    blocks->planes->blocks are identities for k in {5120, 6144, 17408}."""
    rng = np.random.default_rng(11)
    for fmt, nb in [("PQ2_0_G128", 34), ("PTQ1_0_G128", 28)]:
        fmtinfo = oracle.FORMATS[fmt]
        sl = [s for s in oracle.ternary.BLOCK_PLANE_SLICES[fmt] if s is not None]
        assert sum(b - a for a, b in sl) == nb
        assert sorted(i for a, b in sl for i in range(a, b)) == list(range(nb))
        base_s, high_s, _ = oracle.ternary.BLOCK_PLANE_SLICES[fmt]
        assert base_s[1] - base_s[0] == fmtinfo.base_bytes
        assert (0 if high_s is None else high_s[1] - high_s[0]) == fmtinfo.high_bytes
        for k in (5120, 6144, 17408):
            n = 3
            g = oracle.row_split_geometry(fmt, n, k)
            blocks = rng.integers(0, 256, size=n * g.groups_per_row * nb, dtype=np.uint8)
            payload = oracle.blocks_to_planes(fmt, n, k, blocks)
            assert np.array_equal(oracle.planes_to_blocks(fmt, n, k, payload), blocks)
            c = synth.make_case("tiny", n=n, k=k, seed=k)
            p2 = oracle.pack_planes(fmt, c.values, c.scales)
            assert np.array_equal(oracle.blocks_to_planes(fmt, n, k, oracle.planes_to_blocks(fmt, n, k, p2)), p2)


# --------------------------------------------------------------- transform ---
def pin_hadamard_library():
    """The oracle's H equals scipy's Sylvester-construction Hadamard matrix,
    and H @ H = 1024 I."""
    H = oracle.hadamard_matrix(1024)
    assert np.array_equal(H, scipy.linalg.hadamard(1024).astype(np.float64))
    assert np.array_equal(H @ H, 1024.0 * np.eye(1024))


def _fwht(v):
    """Textbook in-place fast Walsh-Hadamard butterfly (natural order)."""
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < v.shape[-1]:
        for i in range(0, v.shape[-1], 2 * h):
            a = v[..., i:i + h].copy()
            b = v[..., i + h:i + 2 * h].copy()
            v[..., i:i + h] = a + b
            v[..., i + h:i + 2 * h] = a - b
        h *= 2
    return v


def pin_hadamard_fast_transform():
    """Dense oracle == per-block fast butterfly, forward (sign then H) and
    inverse (H then sign), on a 3-block input."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3072))
    D = np.where(rng.integers(0, 2, 3072) == 1, -1.0, 1.0)
    fw = oracle.hadamard_forward(x, D)
    iv = oracle.hadamard_inverse(x, D)
    for b in range(3):
        s = slice(1024 * b, 1024 * (b + 1))
        assert np.allclose(fw[:, s], _fwht(D[s] * x[:, s]) / 32, rtol=0, atol=1e-12)
        assert np.allclose(iv[:, s], D[s] * _fwht(x[:, s]) / 32, rtol=0, atol=1e-12)


def pin_hadamard_identities():
    """fwd o inv = inv o fwd = id; l2 norm preserved; blocks independent."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5120))
    D = np.where(rng.integers(0, 2, 5120) == 1, -1.0, 1.0)
    fw = oracle.hadamard_forward(x, D)
    assert np.allclose(oracle.hadamard_inverse(fw, D), x, rtol=0, atol=1e-12)
    assert np.allclose(oracle.hadamard_forward(oracle.hadamard_inverse(x, D), D), x, rtol=0, atol=1e-12)
    assert np.allclose(np.linalg.norm(fw, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    for b in range(5):
        s = slice(1024 * b, 1024 * (b + 1))
        assert np.allclose(np.linalg.norm(fw[:, s], axis=1), np.linalg.norm(x[:, s], axis=1), rtol=1e-13)
    y = x.copy()
    y[:, 2048:3072] += 1.0
    fy = oracle.hadamard_forward(y, D)
    assert np.array_equal(fy[:, :2048], fw[:, :2048]) and np.array_equal(fy[:, 3072:], fw[:, 3072:])


def pin_hadamard_closed_forms():
    """Delta at global position p -> D_p * H[:, p mod 1024] / 32 in p's block
    (forward) and D_j * H[j, p mod 1024] / 32 (inverse); all-ones with D = +1
    -> 32 * e_0 in every block."""
    Hs = scipy.linalg.hadamard(1024).astype(np.float64)
    rng = np.random.default_rng(9)
    D = np.where(rng.integers(0, 2, 2048) == 1, -1.0, 1.0)
    for p in (0, 1, 5, 513, 1023, 1024, 1025, 1500, 2047):
        e = np.zeros((1, 2048))
        e[0, p] = 1.0
        blk, i = divmod(p, 1024)
        s = slice(1024 * blk, 1024 * (blk + 1))
        want_f = np.zeros(2048)
        want_f[s] = D[p] * Hs[:, i] / 32
        want_i = np.zeros(2048)
        want_i[s] = D[s] * Hs[:, i] / 32
        assert np.array_equal(oracle.hadamard_forward(e, D)[0], want_f)
        assert np.array_equal(oracle.hadamard_inverse(e, D)[0], want_i)
    ones = np.ones((1, 2048))
    want = np.zeros(2048)
    want[[0, 1024]] = 32.0
    assert np.array_equal(oracle.hadamard_forward(ones, np.ones(2048))[0], want)


# --------------------------------------------------------------- projection ---
def pin_matmul_library():
    """oracle matmul (pack -> planes -> decode -> transform -> contract) equals
    numpy's matmul of the generator's dense values*scales against x rotated
    with scipy's Hadamard matrix, for both formats and several shapes."""
    Hs = scipy.linalg.hadamard(1024).astype(np.float64)
    for fmt, n, k, M in [("PQ2_0_G128", 37, 2048, 3), ("PTQ1_0_G128", 29, 3072, 2),
                         ("PQ2_0_G128", 256, 1024, 1)]:
        c = synth.make_case("tiny", n=n, k=k, M=M, seed=n + k)
        payload = oracle.pack_planes(fmt, c.values, c.scales)
        y = oracle.ternary_matmul(fmt, payload, n, k, c.x, synth.bf16_bits_to_f32(c.signs))
        D = synth.bf16_bits_to_f32(c.signs).astype(np.float64)
        xr = (c.x.astype(np.float64) * D).reshape(M, k // 1024, 1024) @ Hs.T / 32
        s = np.repeat(c.scales.view(np.float16).astype(np.float64), 128, axis=1)[:, :k]
        want = xr.reshape(M, k) @ (c.values.astype(np.float64) * s).T
        assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
        # row subsets match the full result
        rows = np.array([0, n // 2, n - 1])
        assert np.allclose(oracle.ternary_matmul(fmt, payload, n, k, c.x, D, rows=rows), y[:, rows],
                           rtol=1e-13, atol=1e-13)


def pin_matmul_closed_form():
    """All weights +1, scale 1: y_r = sum_c xr_c = 32 * sum_b D[1024 b] x[1024 b]
    (column sums of H vanish except the first)."""
    rng = np.random.default_rng(21)
    for fmt in ("PQ2_0_G128", "PTQ1_0_G128"):
        n, k = 5, 3072
        values = np.ones((n, k), np.int8)
        scales = np.full((n, k // 128), 0x3C00, np.uint16)
        payload = oracle.pack_planes(fmt, values, scales)
        x = rng.standard_normal((2, k))
        D = np.where(rng.integers(0, 2, k) == 1, -1.0, 1.0)
        y = oracle.ternary_matmul(fmt, payload, n, k, x, D)
        want = 32 * (D[[0, 1024, 2048]] * x[:, [0, 1024, 2048]]).sum(axis=1)
        assert np.allclose(y, want[:, None] * np.ones((1, n)), rtol=1e-12, atol=1e-12)


def pin_matmul_brute_force():
    """Tiny case in pure-Python loops straight from the definitions: every
    weight read from the payload bytes, every product summed one by one."""
    Hs = scipy.linalg.hadamard(1024)
    for fmt in ("PQ2_0_G128", "PTQ1_0_G128"):
        n, k, M = 3, 1024, 2
        c = synth.make_case("tiny", n=n, k=k, M=M, seed=77)
        payload = oracle.pack_planes(fmt, c.values, c.scales)
        D = [1.0 if s == 0x3F80 else -1.0 for s in c.signs]
        g = oracle.row_split_geometry(fmt, n, k)
        y = np.zeros((M, n))
        for m in range(M):
            # rotated input from scipy's Hadamard matrix (a library routine)
            xr = list(Hs @ (np.array(D) * c.x[m].astype(np.float64)) / 32)
            for r in range(n):
                acc = 0.0
                for col in range(k):
                    grp, j = divmod(col, 128)
                    if fmt == "PQ2_0_G128":
                        byte = payload[g.base_offset + r * g.base_row_bytes + grp * 32 + j // 4]
                        val = ((int(byte) >> (2 * (j % 4))) & 3) - 1
                    elif j < 120:
                        byte = int(payload[g.base_offset + r * g.base_row_bytes + grp * 24 + j // 5])
                        val = (byte // 3 ** (j % 5)) % 3 - 1
                    else:
                        byte = int(payload[g.high_offset + r * g.high_row_bytes + grp * 2 + (j - 120) // 4])
                        val = (byte // 3 ** ((j - 120) % 4)) % 3 - 1
                    lo = payload[g.scale_offset + r * g.scale_row_bytes + 2 * grp]
                    hi = payload[g.scale_offset + r * g.scale_row_bytes + 2 * grp + 1]
                    scale = float(np.array([int(lo) | (int(hi) << 8)], np.uint16).view(np.float16)[0])
                    acc += val * scale * xr[col]
                y[m, r] = acc
        got = oracle.ternary_matmul(fmt, payload, n, k, c.x, D)
        assert np.allclose(got, y, rtol=1e-12, atol=1e-12)


def pin_embed_closed_form():
    """Embedding rows: out_i = D * H e_row / 32 per block; with all weights +1,
    scale 1: each block's output is 32 * D * e_0 (H row sums vanish except the first)."""
    rng = np.random.default_rng(8)
    n, k = 6, 2048
    values = np.ones((n, k), np.int8)
    values[3] = -1
    scales = np.full((n, k // 128), 0x3C00, np.uint16)
    payload = oracle.pack_planes("PQ2_0_G128", values, scales)
    D = np.where(rng.integers(0, 2, k) == 1, -1.0, 1.0)
    out = oracle.embed_rows("PQ2_0_G128", payload, n, k, [2, 3, 2], D)
    want = np.zeros((3, k))
    want[:, [0, 1024]] = 32 * D[[0, 1024]]
    want[1] *= -1
    assert np.array_equal(out, want)
    # and the inverse transform undoes the forward one on gathered rows
    c = synth.make_case("tiny", n=50, k=2048, seed=12)
    p2 = oracle.pack_planes("PTQ1_0_G128", c.values, c.scales)
    Ds = synth.bf16_bits_to_f32(c.signs)
    ids = [0, 49, 7, 7]
    out = oracle.embed_rows("PTQ1_0_G128", p2, 50, 2048, ids, Ds)
    W = oracle.dequantize("PTQ1_0_G128", p2, 50, 2048, ids)
    assert np.allclose(oracle.hadamard_forward(out, Ds), W, rtol=0, atol=1e-14)


def pin_padding_bytes():
    """k not a multiple of 128: the pad weights of each row's last group encode
    value 0 (PQ2_0 field 01, PTQ1_0 digit 1), read straight from the bytes."""
    v = np.ones((2, 130), np.int8)
    s = np.full((2, 2), 0x3C00, np.uint16)
    p = oracle.pack_planes("PQ2_0_G128", v, s)
    # row 0, group 1 holds weights 128, 129 (value +1 -> field 10) then 126 pads (01)
    assert p[32] == 0b01011010 and np.all(p[33:64] == 0x55)
    t = oracle.pack_planes("PTQ1_0_G128", v, s)
    # PTQ1_0 row 0 group 1: first base byte = 2 + 2*3 + 1*9 + 1*27 + 1*81 = 125, rest 121; high 40
    assert t[24] == 125 and np.all(t[25:48] == 121)
    g = oracle.row_split_geometry("PTQ1_0_G128", 2, 130)
    assert np.all(t[g.high_offset + 2:g.high_offset + 4] == 40)


def pin_gate_up_limits():
    """SwiGLU of the gate and up projections at points where silu has a closed
    limit: silu(a) -> a for large a, -> 0 for large -a, silu(0) = 0. With x a
    unit vector and every weight +1 the projections are the scales themselves
    (no rotation), or 32 * D[0] * scale (rotation: H's first column is all ones),
    which also tells whether each projection used its own sign vector."""
    n, k = 3, 1024
    ones = np.ones((n, k), np.int8)
    def payload(scale_f16):
        return oracle.pack_planes("PQ2_0_G128", ones, np.full((n, k // 128), scale_f16, np.uint16))
    x = np.zeros((1, k))
    x[0, 0] = 1.0             # unrotated: only column 0 contributes, g = scale
    f16 = lambda v: int(np.array([v], np.float16).view(np.uint16)[0])
    y = oracle.gate_up_swiglu("PQ2_0_G128", payload(f16(20.0)), payload(f16(0.5)), n, k, x)
    assert np.allclose(y, 10.0, rtol=1e-7)                 # silu(20) * 0.5 = 10 (1 - 2e-9)
    y = oracle.gate_up_swiglu("PQ2_0_G128", payload(f16(-20.0)), payload(f16(0.5)), n, k, x)
    assert np.all(np.abs(y) < 1e-6)                        # silu(-20) * 0.5 ~ -2e-8
    y = oracle.gate_up_swiglu("PQ2_0_G128", payload(0), payload(f16(3.0)), n, k, x)
    assert np.all(y == 0.0)                                # silu(0) = 0
    # rotation with different signs: xr = D[0] / 32 everywhere, g = 32 D_g[0] s_g, u = 32 D_u[0] s_u
    Dg = np.ones(k)
    Du = np.ones(k)
    Du[0] = -1.0
    x1 = np.zeros((1, k))
    x1[0, 0] = 1.0
    y = oracle.gate_up_swiglu("PQ2_0_G128", payload(f16(1.0)), payload(f16(1.0 / 32)), n, k, x1, Dg, Du)
    assert np.allclose(y, -32.0, rtol=1e-7)                # silu(32) * (-1)


def pin_ptq1_0_every_byte_value():
    """Every byte value 0..255 of a base and of a high byte decodes to its low
    five (base) or four (high) base-3 digits minus one, the reading that also
    covers bytes the packer never writes. The digits come from numpy's own
    radix conversion (np.base_repr), independent of the oracle's arithmetic."""
    n = 256
    g = oracle.row_split_geometry("PTQ1_0_G128", n, 128)
    payload = np.zeros(g.payload_bytes, np.uint8)
    base = np.full((n, 24), 121, np.uint8)                # 121 = digits 1,1,1,1,1: value 0
    base[:, 7] = np.arange(n)                              # weights 35 .. 39
    high = np.full((n, 2), 40, np.uint8)                   # 40 = digits 1,1,1,1
    high[:, 1] = np.arange(n)                              # weights 124 .. 127
    payload[:g.base_bytes] = base.reshape(-1)
    payload[g.high_offset:g.high_offset + g.high_bytes] = high.reshape(-1)
    payload[g.scale_offset:] = np.tile(np.array([0, 0x3C], np.uint8), n)     # scale 1.0
    W = oracle.dequantize("PTQ1_0_G128", payload, n, 128)

    def digits(B, count):
        r = np.base_repr(int(B), base=3)[::-1] + "0" * 8
        return [int(ch) for ch in r[:count]]

    for B in range(n):
        assert list(W[B, 35:40]) == [d - 1 for d in digits(B, 5)], B
        assert list(W[B, 124:128]) == [d - 1 for d in digits(B, 4)], B
        assert np.all(W[B, :35] == 0) and np.all(W[B, 40:124] == 0)


# ----------------------------------------------------------- error figures ---
def pin_max_rel_error_worked():
    """The infinity-norm relative error on hand-worked vectors. Each case is
    chosen so that one plausible slip changes the answer: a dropped absolute
    value (a negative largest difference), the denominator taken from got
    instead of ref (max |got| > max |ref|), a mean in place of a max, and the
    all-zero reference convention (absolute error)."""
    f = oracle.max_rel_error
    # |3 - 4| / 4: the largest difference is negative
    assert f([1.0, 2.0, 3.0], [1.0, 2.0, 4.0]) == 0.25
    # |5 - 4| / 4 = 0.25 as well (sign of the difference does not matter)
    assert f([1.0, 2.0, 5.0], [1.0, 2.0, 4.0]) == 0.25
    # max |got| = 8 > max |ref| = 4: normalised by the reference, 4 / 4 = 1
    assert f([0.0, 0.0, 8.0], [0.0, 0.0, 4.0]) == 1.0
    # largest difference (0.5 at index 0) and largest |ref| (-10 at index 2) differ
    assert f([1.5, -3.0, -10.0], [1.0, -3.0, -10.0]) == 0.05
    # 2-D arrays are compared element by element, whole-array maxima
    assert f(np.array([[1.0, 2.0], [3.0, 4.5]]), np.array([[1.0, 2.0], [3.0, 4.0]])) == 0.125
    # all-zero reference: the absolute error; identical zero vectors score 0
    assert f([0.5, 0.0], [0.0, 0.0]) == 0.5
    assert f([0.0, -0.25], [0.0, 0.0]) == 0.25
    assert f([0.0, 0.0], [0.0, 0.0]) == 0.0
    # identical vectors score exactly 0
    assert f([3.0, -7.0, 1e-300], [3.0, -7.0, 1e-300]) == 0.0


def pin_significant_rel_error_worked():
    """The per-element relative error over |ref_i| >= 0.1 * rms(ref), on
    hand-worked vectors. ref = (10, 0.8, 0.01, -5): rms = sqrt(125.6401 / 4)
    = 5.6045.., so the threshold 0.56 keeps 10, 0.8 and -5 and drops 0.01
    (a threshold of 0.1 * max = 1.0 would also drop 0.8)."""
    f = oracle.significant_rel_error
    ref = [10.0, 0.8, 0.01, -5.0]
    # errors 0.1/10, 0.04/0.8, (0.49/0.01 dropped), 0.2/5 -> 0.05 from the 0.8 element
    assert abs(f([10.1, 0.84, 0.5, -5.2], ref) - 0.05) < 1e-12
    # the small element alone is wrong: it is below the threshold, so 0
    assert f([10.0, 0.8, 0.5, -5.0], ref) == 0.0
    # negative reference element, got on the far side of zero: |-4 - (-5)| / 5 = 0.2
    assert abs(f([10.0, 0.8, 0.01, -4.0], ref) - 0.2) < 1e-12
    # relative to |ref_i| (0.8), not to max |ref|: 0.4 / 0.8 = 0.5
    assert abs(f([10.0, 1.2, 0.01, -5.0], ref) - 0.5) < 1e-12
    # all elements equal in size: every one qualifies, 1/2
    assert f([1.0, -1.0, 1.5], [1.0, -1.0, 1.0]) == 0.5
    # empty and all-zero references
    assert f([], []) == 0.0 and f([0.3, 0.0], [0.0, 0.0]) == 0.0
    # a different floor: 0.5 * rms = 2.80 keeps only 10 and -5
    assert abs(f([10.1, 1.2, 0.01, -5.2], ref, floor=0.5) - 0.04) < 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
