"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small shapes span several tiles and ragged tails and compare every output;
the full-size workloads compare all outputs where the oracle finishes in
seconds and sampled rows otherwise. Tolerance (infinity-norm relative error,
max|y - y_ref| / max|y_ref|): 1e-3 for the decode projection, the transform
and the embedding; 2e-2 for the 16-bit tensor-core prefill path. The
projections and the embedding also bound the per-element relative error over
the outputs that are not small (|y_ref| >= 0.1 rms(y_ref)): 1e-2 and 2e-2.
"""
import numpy as np
import pytest
import torch

import bit_gemv_gb300 as nt
import oracle
import synth
from gpu_util import DEV, dev_signs, dev_u8, dev_x, oracle_matmul_rows, run_matmul, signs_values

pytestmark = pytest.mark.gpu

TOL_DECODE = 1e-3
TOL_PREFILL = 2e-2
# Per-element relative error over the outputs with |y_ref| >= 0.1 rms(y_ref).
# The decode kernels round the rotated activation to 16 bits (integer path:
# 14-bit magnitude per 1024-block; MMA path: binary16), which leaves an output
# error of about 1e-4 rms(y); at 0.1 rms(y) that is a per-element error near
# 1e-3 rms and a few times that at the maximum over ~1e4 such outputs. The
# bounds below keep a margin of about three over that estimate.
TOL_DECODE_ELEM = 1e-2
TOL_PREFILL_ELEM = 2e-2


def check_decode(y, ref):
    """Both accuracy figures for a decode, transform or embedding result."""
    e, s = oracle.max_rel_error(y, ref), oracle.significant_rel_error(y, ref)
    assert e <= TOL_DECODE and s <= TOL_DECODE_ELEM, (e, s)


def check_prefill(y, ref):
    """Both accuracy figures for a tensor-core prefill result."""
    e, s = oracle.max_rel_error(y, ref), oracle.significant_rel_error(y, ref)
    assert e <= TOL_PREFILL and s <= TOL_PREFILL_ELEM, (e, s)


# ---------------------------------------------------------------- transform ---
@pytest.mark.parametrize("x_dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("y_dtype", [torch.float32, torch.bfloat16])
def test_hadamard_forward_inverse(x_dtype, y_dtype):
    rng = np.random.default_rng(10)
    M, K = 5, 3072
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(DEV).to(x_dtype)
    sbits = synth.sign_vector(rng, K)
    s = dev_signs(sbits)
    D = synth.bf16_bits_to_f32(sbits)
    xv = x.float().cpu().numpy().astype(np.float64)
    fw = nt.ninfer_hadamard_fwd(x, s, out_dtype=y_dtype)
    iv = nt.ninfer_hadamard_inv(x, s, out_dtype=y_dtype)
    torch.cuda.synchronize()
    tol = 1e-5 if y_dtype == torch.float32 else 4e-3
    assert oracle.max_rel_error(fw.float().cpu().numpy(), oracle.hadamard_forward(xv, D)) <= tol
    assert oracle.max_rel_error(iv.float().cpu().numpy(), oracle.hadamard_inverse(xv, D)) <= tol


def test_hadamard_in_place_and_roundtrip():
    rng = np.random.default_rng(11)
    M, K = 3, 17408
    x0 = rng.standard_normal((M, K)).astype(np.float32)
    sbits = synth.sign_vector(rng, K)
    s = dev_signs(sbits)
    x = torch.from_numpy(x0).to(DEV)
    nt.ninfer_hadamard_fwd(x, s, out=x)            # in place
    ref = oracle.hadamard_forward(x0, synth.bf16_bits_to_f32(sbits))
    assert oracle.max_rel_error(x.cpu().numpy(), ref) <= 1e-5
    nt.ninfer_hadamard_inv(x, s, out=x)
    assert oracle.max_rel_error(x.cpu().numpy(), x0) <= 1e-5


# ------------------------------------------------------------------ matmul ---
def test_matmul_tiny_workload():
    c = synth.make_case("tiny")
    y = run_matmul("PQ2_0_G128", c)
    ref = oracle_matmul_rows("PQ2_0_G128", c, np.arange(c.workload.n))
    check_decode(y, ref)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("n,k,M", [(300, 2048, 1), (300, 2048, 8), (77, 3072, 3), (1, 1024, 1), (17, 5120, 2),
                                   (1000, 1024, 5), (31, 2048, 1), (517, 5120, 1), (50001, 1024, 1),
                                   (150, 2048, 1), (80, 2048, 1), (150, 2048, 4)])
def test_matmul_small_shapes(fmt, n, k, M):
    c = synth.make_case("gateup", n=n, k=k, M=M, seed=n * 7 + k + M)
    y = run_matmul(fmt, c)
    ref = oracle_matmul_rows(fmt, c, np.arange(n))
    check_decode(y, ref)


@pytest.mark.parametrize("n,k,M", [(4099, 3072, 7), (2100, 2048, 8), (63, 9216, 4), (16, 1024, 2)])
def test_matmul_ptq1_block_split(n, k, M):
    """PTQ1_0 with 2 <= M <= 8: the CTA grid is 1024-blocks x row tiles (each
    tile a multiple of 16 rows, the last one ragged) and the per-block partial
    sums are added by a second kernel; n % 4 != 0 pads the partial rows."""
    c = synth.make_case("down", n=n, k=k, M=M, seed=n + k + M)
    y = run_matmul("PTQ1_0_G128", c)
    ref = oracle_matmul_rows("PTQ1_0_G128", c, np.arange(n))
    check_decode(y, ref)


@pytest.mark.parametrize("n,k,rotate", [(40, 16384, True), (300, 17408, True), (200, 32768, True),
                                        (150, 34816, True), (90, 33700, False), (70, 20400, False)])
def test_matmul_ptq1_m1_wide_k(n, k, rotate):
    """PTQ1_0 at M = 1 with 16 to 34 1024-blocks (rotated, and raw with a
    ragged last block): clusters of two or four CTAs split the groups, each CTA
    rotating only the blocks of its share, and add their row sums through
    distributed shared memory."""
    c = synth.make_case("down", n=n, k=k, M=1, seed=n + k)
    y = run_matmul("PTQ1_0_G128", c, rotate=rotate)
    ref = oracle_matmul_rows("PTQ1_0_G128", c, np.arange(n), rotate=rotate)
    check_decode(y, ref)


@pytest.mark.parametrize("n,k", [(200, 8192), (200, 9216), (200, 16384), (200, 17408), (90, 19456), (20000, 17408),
                                 (3, 73728), (700, 69632), (64, 147456)])
def test_matmul_ptq1_m1_group_split(n, k):
    """PTQ1_0 at M = 1 around the group split: eight blocks (one CTA's eight
    warp pairs rotate them in one round), nine and sixteen (a cluster of two
    CTAs, each rotating and reading its half), seventeen and nineteen (four
    CTAs with 34 and 38 groups each, so that the high-byte and scale segments of
    neighbouring ranks are rounded out to whole 16-byte units and overlap), a
    ring refilled many times per cluster (n = 20000), and 144 to 288 groups per
    CTA (several rotation rounds, one to three row sets)."""
    c = synth.make_case("down", n=n, k=k, M=1, seed=n + 3 * k)
    y = run_matmul("PTQ1_0_G128", c)
    if n > 1000:
        rows = np.unique(np.concatenate([np.arange(0, n, 97), [n - 1], np.arange(250, 300)]))
    else:
        rows = np.arange(n)
    ref = oracle_matmul_rows("PTQ1_0_G128", c, rows)
    check_decode(y[:, rows] if n > 1000 else y, ref)


@pytest.mark.parametrize("n,k,rotate", [(300, 16384, True), (130, 20480, True), (90, 20400, False),
                                        (200, 8192, True), (4800, 9216, True)])
def test_matmul_pq2_m1_wide_k(n, k, rotate):
    """PQ2_0 at M = 1 with more than seven 1024-blocks: CTA pairs (clusters)
    share the rotations, a warp pair rotating one block per round; an odd
    number of CTAs with rows (n = 200: three, n = 4800: seventy-five) adds a
    CTA without rows that only rotates for its partner."""
    c = synth.make_case("gateup", n=n, k=k, M=1, seed=n + k)
    y = run_matmul("PQ2_0_G128", c, rotate=rotate)
    ref = oracle_matmul_rows("PQ2_0_G128", c, np.arange(n), rotate=rotate)
    check_decode(y, ref)


@pytest.mark.slow
def test_matmul_ptq1_ring_refill():
    """Row tiles longer than the shared-memory ring (more than six items of 128
    rows per CTA at k = 17408): slots are released and refilled mid-tile.
    Sampled rows from every tile."""
    c = synth.make_case("down", n=8000, k=17408, M=3, seed=44)
    y = run_matmul("PTQ1_0_G128", c)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(0, 8000, 97), [7999], rng.integers(0, 8000, 400)]))
    ref = oracle_matmul_rows("PTQ1_0_G128", c, rows)
    check_decode(y[:, rows], ref)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("n,k,M", [(70, 1000, 4), (40, 1001, 3), (33, 2040, 1)])
def test_matmul_unrotated_ragged_k(fmt, n, k, M):
    """Raw input with k just under a multiple of 1024: the decode kernels take
    k = 1000 and 2040 (x rows stay 16-byte aligned, the missing elements of the
    last block are zero); k = 1001 leaves the rows of x unaligned and must be
    served by the general path."""
    c = synth.make_case("gateup", n=n, k=k, M=M, seed=n + k)
    y = run_matmul(fmt, c, rotate=False)
    ref = oracle_matmul_rows(fmt, c, np.arange(n), rotate=False)
    check_decode(y, ref)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_matmul_unrotated_padded_k(fmt):
    """No hadamard_signs (raw input) and k % 128 != 0: the pad columns of the
    last group must not contribute."""
    c = synth.make_case("gateup", n=129, k=300, M=2, seed=5)
    y = run_matmul(fmt, c, rotate=False)
    ref = oracle_matmul_rows(fmt, c, np.arange(129), rotate=False)
    check_decode(y, ref)


def test_matmul_bf16_output():
    c = synth.make_case("gateup", n=512, k=5120, M=1, seed=9)
    y = run_matmul("PQ2_0_G128", c, y_dtype=torch.bfloat16)
    ref = oracle_matmul_rows("PQ2_0_G128", c, np.arange(512))
    assert oracle.max_rel_error(y, ref) <= 4e-3       # bf16 output rounding


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("n,k", [(300, 5120), (200, 17408)])
@pytest.mark.parametrize("x_dtype,y_dtype", [(torch.float32, torch.float32), (torch.float16, torch.float32),
                                             (torch.float16, torch.bfloat16), (torch.float32, torch.bfloat16)])
def test_matmul_m1_activation_and_output_dtypes(fmt, n, k, x_dtype, y_dtype):
    """The M = 1 kernels for every activation dtype (each is a separate
    instance) and bf16 outputs, also through the exchange of the clustered
    PTQ1_0 path (k = 17408: clusters of four CTAs). The oracle takes the
    activation as the kernel sees it (rounded to the input dtype)."""
    c = synth.make_case("gateup", n=n, k=k, M=1, seed=n + k + 7)
    xd = torch.from_numpy(c.x.astype(np.float32)).to(DEV).to(x_dtype)
    payload = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    y = nt.ninfer_ternary_matmul(fmt, payload, n, k, xd, dev_signs(c.signs), y_dtype=y_dtype)
    torch.cuda.synchronize()
    xs = xd.float().cpu().numpy().astype(np.float64)
    ref = oracle.ternary_matmul(fmt, oracle.pack_planes(fmt, c.values, c.scales), n, k, xs, signs_values(c))
    got = y.float().cpu().numpy().astype(np.float64)
    if y_dtype == torch.float32:
        check_decode(got, ref)
    else:
        assert oracle.max_rel_error(got, ref) <= 4e-3      # bf16 output rounding


@pytest.mark.slow
def test_matmul_gateup_full():
    c = synth.make_case("gateup")
    y = run_matmul("PQ2_0_G128", c)
    ref = oracle_matmul_rows("PQ2_0_G128", c, np.arange(c.workload.n))
    check_decode(y, ref)


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 8])
def test_matmul_down_full(M):
    c = synth.make_case("down", M=M)
    y = run_matmul("PTQ1_0_G128", c)
    ref = oracle_matmul_rows("PTQ1_0_G128", c, np.arange(c.workload.n))
    check_decode(y, ref)


@pytest.fixture(scope="module")
def head_case():
    """The output-head matrix (248320 x 5120, seed 4) with 8 activation rows and
    64 token ids; its payload is packed per format on first use (PQ2_0:
    337,715,200 bytes; PTQ1_0: 278,118,400 bytes), one format on the device at
    a time."""
    c = synth.make_case("head", M=8, with_ids=True)
    cache = {}

    def payload(fmt):
        if fmt not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[fmt] = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
        return cache[fmt]
    return c, payload


HEAD_FORMATS = ["PQ2_0_G128", "PTQ1_0_G128"]


@pytest.mark.slow
@pytest.mark.parametrize("fmt", HEAD_FORMATS)
@pytest.mark.parametrize("M", [1, 8])
def test_matmul_head_sampled(head_case, fmt, M):
    """The head shape in both formats: over 1,600 rows per CTA at M = 1 (PQ2_0 and
    PTQ1_0 rings refilled many times per CTA), sampled rows (the first, the
    last, 3,000 random) against the oracle, which packs exactly those rows."""
    c, payload = head_case
    sub = synth.Case(c.workload, c.values, c.scales, c.signs, c.x[:M], c.x_raw[:M])
    y = run_matmul(fmt, sub, payload_dev=payload(fmt))
    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, 1, c.workload.n - 1], rng.integers(0, c.workload.n, 3000)]))
    ref = oracle_matmul_rows(fmt, sub, rows)
    check_decode(y[:, rows], ref)
    assert np.all(np.isfinite(y))


@pytest.mark.slow
@pytest.mark.parametrize("fmt", HEAD_FORMATS)
def test_embed_head_rows(head_case, fmt):
    c, payload = head_case
    n, k = c.values.shape
    ids = torch.from_numpy(c.ids).to(DEV)
    out = nt.ninfer_ternary_embed(fmt, payload(fmt), n, k, ids, dev_signs(c.signs))
    torch.cuda.synchronize()
    sub = oracle.pack_planes(fmt, c.values[c.ids], c.scales[c.ids])
    ref = oracle.embed_rows(fmt, sub, c.ids.size, k, np.arange(c.ids.size), signs_values(c))
    check_decode(out.cpu().numpy(), ref)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("preset,n,k,M", [("prefill", 300, 1024, 200), ("prefill", 129, 2048, 130),
                                           ("tiny", 256, 1024, 17), ("prefill", 1000, 5120, 300)])
def test_matmul_prefill_small(fmt, preset, n, k, M):
    """Tensor-core prefill path: partial token and weight-row tiles, fp32 and
    bf16 activations, every output compared. PTQ1_0 runs through its planes
    rewritten as PQ2_0 planes on the device."""
    c = synth.make_case(preset, n=n, k=k, M=M, seed=n + k + M)
    y = run_matmul(fmt, c)
    ref = oracle_matmul_rows(fmt, c, np.arange(n))
    check_prefill(y, ref)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_matmul_prefill_multi_tile(fmt):
    """60 x 8 output tiles (the last of each ragged) on one persistent CTA per
    SM: every CTA walks three or four tiles, so both tensor-memory accumulator
    buffers are reused and handed back by the epilogue. Every output compared."""
    c = synth.make_case("prefill", n=7601, k=1024, M=1500, seed=7)
    y = run_matmul(fmt, c)
    ref = oracle_matmul_rows(fmt, c, np.arange(7601))
    check_prefill(y, ref)


def test_matmul_prefill_ptq1_invalid_trits():
    """Base bytes >= 243 and high bytes >= 81 are not produced by the packer;
    every decoder follows the digit definition (byte / 3^i) % 3 for them too, so
    the rewritten PQ2_0 planes must give the oracle's result on such payloads."""
    c = synth.make_case("prefill", n=40, k=1024, M=24, seed=77)
    payload = nt.ninfer_ternary_pack("PTQ1_0_G128", c.values, c.scales)
    g = nt.ninfer_ternary_geometry("PTQ1_0_G128", 40, 1024)
    rng = np.random.default_rng(3)
    pay = payload.copy()
    base = pay[g.base_offset:g.base_offset + g.base_bytes]
    high = pay[g.high_offset:g.high_offset + g.high_bytes]
    base[rng.integers(0, base.size, 60)] = rng.integers(243, 256, 60).astype(np.uint8)
    high[rng.integers(0, high.size, 20)] = rng.integers(81, 256, 20).astype(np.uint8)
    y = run_matmul("PTQ1_0_G128", c, payload_dev=dev_u8(pay))
    ref = oracle.ternary_matmul("PTQ1_0_G128", pay, 40, 1024, c.x, signs_values(c))
    check_prefill(y, ref)


def test_matmul_prefill_unrotated_bf16_out():
    c = synth.make_case("prefill", n=256, k=2048, M=64, seed=11)
    y = run_matmul("PQ2_0_G128", c, rotate=False, y_dtype=torch.bfloat16)
    ref = oracle_matmul_rows("PQ2_0_G128", c, np.arange(256), rotate=False)
    check_prefill(y, ref)


@pytest.mark.slow
def test_matmul_prefill_down_sampled():
    c = synth.make_case("prefill_down")
    y = run_matmul("PTQ1_0_G128", c)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, c.workload.n - 1], rng.integers(0, c.workload.n, 128)]))
    ref = oracle_matmul_rows("PTQ1_0_G128", c, rows)
    check_prefill(y[:, rows], ref)


@pytest.mark.slow
def test_matmul_prefill_sampled():
    c = synth.make_case("prefill")
    y = run_matmul("PQ2_0_G128", c)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, c.workload.n - 1], rng.integers(0, c.workload.n, 256)]))
    ref = oracle_matmul_rows("PQ2_0_G128", c, rows)
    check_prefill(y[:, rows], ref)


# --------------------------------------------------------------- embedding ---
@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_embed_small(fmt):
    c = synth.make_case("gateup", n=500, k=3072, M=1, seed=21)
    payload = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    ids_np = np.array([0, 499, 7, 7, 250], np.int32)
    out = nt.ninfer_ternary_embed(fmt, payload, 500, 3072, torch.from_numpy(ids_np).to(DEV), dev_signs(c.signs))
    torch.cuda.synchronize()
    ref = oracle.embed_rows(fmt, oracle.pack_planes(fmt, c.values, c.scales), 500, 3072, ids_np, signs_values(c))
    check_decode(out.cpu().numpy(), ref)


def test_embed_out_of_range_ids_flagged():
    c = synth.make_case("gateup", n=64, k=1024, M=1, seed=22)
    payload = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", c.values, c.scales))
    ids = torch.tensor([3, -1, 64, 5], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = nt.ninfer_ternary_embed("PQ2_0_G128", payload, 64, 1024, ids, dev_signs(c.signs), status=status)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert status.item() == 1
    assert np.all(o[1] == 0) and np.all(o[2] == 0)
    ref = oracle.embed_rows("PQ2_0_G128", oracle.pack_planes("PQ2_0_G128", c.values, c.scales), 64, 1024, [3, 5],
                            signs_values(c))
    check_decode(o[[0, 3]], ref)
    status.zero_()
    nt.ninfer_ternary_embed("PQ2_0_G128", payload, 64, 1024, ids[[0, 3]].contiguous(), dev_signs(c.signs), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0


def test_embed_unrotated():
    c = synth.make_case("gateup", n=40, k=300, M=1, seed=23)
    payload = dev_u8(nt.ninfer_ternary_pack("PTQ1_0_G128", c.values, c.scales))
    ids = torch.tensor([1, 39], dtype=torch.int32, device=DEV)
    out = nt.ninfer_ternary_embed("PTQ1_0_G128", payload, 40, 300, ids)
    torch.cuda.synchronize()
    W = oracle.dequantize("PTQ1_0_G128", oracle.pack_planes("PTQ1_0_G128", c.values, c.scales), 40, 300, [1, 39])
    assert np.array_equal(out.cpu().numpy().astype(np.float64), W)


def test_no_device_errors_after_suite():
    torch.cuda.synchronize()
    assert nt.ninfer_device_errors(clear=True) == 0


@pytest.mark.parametrize("fmt,n,k", [("PQ2_0_G128", 600, 5120), ("PQ2_0_G128", 3000, 16384),
                                     ("PTQ1_0_G128", 600, 5120), ("PTQ1_0_G128", 20000, 17408)])
def test_bounded_wait_failure_path(fmt, n, k):
    """A weight-ring wait that gives up: with the bound set to 0 every wait of
    the M = 1 kernels gives up at its first check, although the copies land
    normally. The call still returns OK and sets bit 0 of the device error word
    (the call's output is not meaningful); the CTAs let their issued copies
    land before exiting, so the context stays usable: the next call with the
    default bound matches the oracle and leaves the word clear. The second and
    fourth shapes have more ring items per CTA than slots; the fourth runs the
    PTQ1_0 kernel in clusters of four CTAs, whose barriers every thread still
    reaches. Output rows are sampled for the large shape."""
    c = synth.make_case("gateup", n=n, k=k, M=1, seed=n + k)
    payload = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    torch.cuda.synchronize()
    assert nt.ninfer_device_errors(clear=True) == 0
    try:
        nt.ninfer_set_wait_limit(0)
        nt.ninfer_ternary_matmul(fmt, payload, n, k, dev_x(c), dev_signs(c.signs))
        torch.cuda.synchronize()
    finally:
        nt.ninfer_set_wait_limit(nt.WAIT_LIMIT_DEFAULT)
    assert nt.ninfer_device_errors(clear=True) & 1
    y = run_matmul(fmt, c, payload_dev=payload)
    rows = np.arange(n) if n <= 3000 else np.unique(np.concatenate([np.arange(0, n, 53), [n - 1]]))
    check_decode(y[:, rows], oracle_matmul_rows(fmt, c, rows))
    assert nt.ninfer_device_errors(clear=True) == 0


# --------------------------------------------------------- block <-> planes ---
@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("n,k", [(1, 128), (37, 1000), (300, 5120)])
def test_blocks_planes_device_matches_oracle(fmt, n, k):
    """Device block-stream <-> plane conversion, bit-exact against the oracle's
    own conversion of the same generator output (both directions)."""
    c = synth.make_case("gateup", n=n, k=k, M=1, seed=n + k)
    payload = oracle.pack_planes(fmt, c.values, c.scales)
    blocks = oracle.planes_to_blocks(fmt, n, k, payload)
    got_payload = nt.ninfer_blocks_to_planes_device(fmt, n, k, dev_u8(blocks))
    got_blocks = nt.ninfer_planes_to_blocks_device(fmt, n, k, dev_u8(payload))
    torch.cuda.synchronize()
    assert np.array_equal(got_payload.cpu().numpy(), oracle.blocks_to_planes(fmt, n, k, blocks))
    assert np.array_equal(got_blocks.cpu().numpy(), blocks)


# ------------------------------------------------------- fused FFN gate/up ---
_up_inputs = synth.up_projection     # the up projection's values, scales and signs, from their own generator


@pytest.mark.parametrize("fmt,n,k,M,same_signs", [
    ("PQ2_0_G128", 300, 2048, 1, False), ("PQ2_0_G128", 300, 2048, 1, True), ("PQ2_0_G128", 150, 5120, 1, False),
    ("PQ2_0_G128", 1, 1024, 1, False), ("PTQ1_0_G128", 300, 2048, 1, False), ("PQ2_0_G128", 77, 3072, 4, False),
    ("PTQ1_0_G128", 129, 2048, 40, True), ("PQ2_0_G128", 200, 5120, 1, False), ("PQ2_0_G128", 4800, 4096, 1, False)])
def test_gate_up_swiglu(fmt, n, k, M, same_signs):
    """silu(gate x) * (up x), each projection with its own signs (or one shared
    vector): PQ2_0 at M = 1 runs the fused two-matrix kernel, the other cases
    the two projections and the SwiGLU kernel."""
    c = synth.make_case("gateup", n=n, k=k, M=M, seed=n + k + M)
    vu, su, du = _up_inputs(n + 2 * k + M, n, k)
    if same_signs:
        du = c.signs
    pay_g = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    pay_u = dev_u8(nt.ninfer_ternary_pack(fmt, vu, su))
    sg = dev_signs(c.signs)
    su_dev = sg if same_signs else dev_signs(du)
    y = nt.ninfer_ternary_gate_up(fmt, pay_g, pay_u, n, k, dev_x(c), sg, su_dev)
    torch.cuda.synchronize()
    ref = oracle.gate_up_swiglu(fmt, oracle.pack_planes(fmt, c.values, c.scales), oracle.pack_planes(fmt, vu, su), n, k,
                                c.x, signs_values(c), synth.bf16_bits_to_f32(du).astype(np.float64))
    tol = TOL_DECODE if M <= 8 else TOL_PREFILL
    assert oracle.max_rel_error(y.cpu().numpy().astype(np.float64), ref) <= tol


def test_gate_up_unrotated_and_errors():
    c = synth.make_case("gateup", n=64, k=1000, M=1, seed=3)
    vu, su, _ = _up_inputs(4, 64, 1000)
    pay_g = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", c.values, c.scales))
    pay_u = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", vu, su))
    y = nt.ninfer_ternary_gate_up("PQ2_0_G128", pay_g, pay_u, 64, 1000, dev_x(c))
    torch.cuda.synchronize()
    ref = oracle.gate_up_swiglu("PQ2_0_G128", oracle.pack_planes("PQ2_0_G128", c.values, c.scales),
                                oracle.pack_planes("PQ2_0_G128", vu, su), 64, 1000, c.x)
    assert oracle.max_rel_error(y.cpu().numpy().astype(np.float64), ref) <= TOL_DECODE
    with pytest.raises(nt.NinferError):          # one sign vector without the other
        nt.ninfer_ternary_gate_up("PQ2_0_G128", pay_g, pay_u, 64, 1024, dev_x(synth.make_case("gateup", n=64, k=1024, M=1, seed=3)),
                                  dev_signs(synth.make_case("gateup", n=64, k=1024, M=1, seed=3).signs), None)


@pytest.mark.slow
def test_gate_up_full_sampled():
    """The gate/up shape (17408 x 5120 per projection), M = 1, fused kernel;
    sampled rows of both projections from the oracle."""
    c = synth.make_case("gateup")
    n, k = c.values.shape
    vu, su, du = _up_inputs(11, n, k)
    pay_g = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", c.values, c.scales))
    pay_u = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", vu, su))
    y = nt.ninfer_ternary_gate_up("PQ2_0_G128", pay_g, pay_u, n, k, dev_x(c), dev_signs(c.signs), dev_signs(du))
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 2000)]))
    ref = oracle.gate_up_swiglu("PQ2_0_G128", oracle.pack_planes("PQ2_0_G128", c.values[rows], c.scales[rows]),
                                oracle.pack_planes("PQ2_0_G128", vu[rows], su[rows]), rows.size, k, c.x,
                                signs_values(c), synth.bf16_bits_to_f32(du).astype(np.float64))
    assert oracle.max_rel_error(y.cpu().numpy()[:, rows].astype(np.float64), ref) <= TOL_DECODE


# ------------------------------------------ chained calls in a CUDA graph ---
def _graph(fn):
    """fn() captured in a CUDA graph on a side stream (as bench.py captures its
    back-to-back calls; each call is launched with programmatic dependent launch
    on the one before)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def test_ffn_chain_graph_replay():
    """The FFN at full size, chained as a decoder runs it: the fused gate/up
    pair with SwiGLU (PQ2_0, 17408 x 5120) writes h in bf16, and the down
    projection (PTQ1_0, 5120 x 17408) reads h as its x. Three tokens run
    eagerly into separate buffers and are checked against the oracle (sampled
    gate/up rows; every down row from the oracle applied to the h the GPU
    produced). The same three chains, captured back to back in one CUDA graph
    with a single shared h buffer (each call waits for the one before it to
    finish reading and writing h), must reproduce the eager outputs bit for
    bit: every kernel adds in a fixed order."""
    cg = synth.make_case("gateup")
    cd = synth.make_case("down")
    n, k = cg.values.shape                      # 17408 x 5120
    nd, kd = cd.values.shape                    # 5120 x 17408
    assert kd == n and nd == k
    vu, su, du = _up_inputs(11, n, k)
    pay_g = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", cg.values, cg.scales))
    pay_u = dev_u8(nt.ninfer_ternary_pack("PQ2_0_G128", vu, su))
    pay_d = dev_u8(nt.ninfer_ternary_pack("PTQ1_0_G128", cd.values, cd.scales))
    sg, su_d, sd = dev_signs(cg.signs), dev_signs(du), dev_signs(cd.signs)
    T = 3
    xv, xraw = synth.activations(np.random.default_rng(21), T, k, "bf16")
    xs = [torch.from_numpy(np.ascontiguousarray(xraw[t:t + 1]).view(np.int16)).to(DEV).view(torch.bfloat16)
          for t in range(T)]

    def chain(h_bufs, y_bufs):
        for t in range(T):
            nt.ninfer_ternary_gate_up("PQ2_0_G128", pay_g, pay_u, n, k, xs[t], sg, su_d, y=h_bufs[t])
            nt.ninfer_ternary_matmul("PTQ1_0_G128", pay_d, nd, kd, h_bufs[t], sd, y=y_bufs[t])

    h_e = [torch.empty((1, n), dtype=torch.bfloat16, device=DEV) for _ in range(T)]
    y_e = [torch.empty((1, nd), dtype=torch.float32, device=DEV) for _ in range(T)]
    chain(h_e, y_e)
    torch.cuda.synchronize()
    h_np = np.concatenate([h.float().cpu().numpy() for h in h_e]).astype(np.float64)
    y_np = np.concatenate([y.cpu().numpy() for y in y_e]).astype(np.float64)

    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(6).integers(0, n, 1500)]))
    ref_h = oracle.gate_up_swiglu("PQ2_0_G128", oracle.pack_planes("PQ2_0_G128", cg.values[rows], cg.scales[rows]),
                                  oracle.pack_planes("PQ2_0_G128", vu[rows], su[rows]), rows.size, k, xv,
                                  signs_values(cg), synth.bf16_bits_to_f32(du).astype(np.float64))
    # h is stored in bf16: compare within bf16 rounding on top of the decode bound
    assert oracle.max_rel_error(h_np[:, rows], ref_h) <= TOL_DECODE + 2.0 ** -8
    ref_y = oracle.ternary_matmul("PTQ1_0_G128", oracle.pack_planes("PTQ1_0_G128", cd.values, cd.scales), nd, kd,
                                  h_np, signs_values(cd))
    check_decode(y_np, ref_y)

    h_shared = torch.empty((1, n), dtype=torch.bfloat16, device=DEV)
    y_g = [torch.full((1, nd), float("nan"), dtype=torch.float32, device=DEV) for _ in range(T)]
    g = _graph(lambda: chain([h_shared] * T, y_g))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(y_g[t], y_e[t]), t
    assert torch.equal(h_shared, h_e[T - 1])
    assert nt.ninfer_device_errors() == 0


def test_gateup_graph_replay_rotating_pool():
    """The gate/up projection (PQ2_0 17408 x 5120, M = 1) as bench.py times it:
    back-to-back calls in a CUDA graph over a rotating pool of payload copies.
    Every call's output equals the eager call's bit for bit, and the eager
    output matches the oracle on sampled rows."""
    c = synth.make_case("gateup")
    n, k = c.values.shape
    host = nt.ninfer_ternary_pack("PQ2_0_G128", c.values, c.scales)
    pool = [dev_u8(host) for _ in range(2)]
    x, s = dev_x(c), dev_signs(c.signs)
    y_ref = nt.ninfer_ternary_matmul("PQ2_0_G128", pool[0], n, k, x, s)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(8).integers(0, n, 1500)]))
    check_decode(y_ref.cpu().numpy()[:, rows].astype(np.float64), oracle_matmul_rows("PQ2_0_G128", c, rows))
    K = 6
    ys = [torch.full((1, n), float("nan"), dtype=torch.float32, device=DEV) for _ in range(K)]
    g = _graph(lambda: [nt.ninfer_ternary_matmul("PQ2_0_G128", pool[i % 2], n, k, x, s, y=ys[i]) for i in range(K)])
    g.replay()
    torch.cuda.synchronize()
    for i in range(K):
        assert torch.equal(ys[i], y_ref), i
    assert nt.ninfer_device_errors() == 0


@pytest.mark.parametrize("fmt,wl", [("PQ2_0_G128", "gateup"), ("PTQ1_0_G128", "down")])
def test_m8_graph_replay_shared_workspace(fmt, wl):
    """M = 8 decode at the full gate/up and down shapes, three calls back to
    back through one shared workspace (PQ2_0: the activation fragments;
    PTQ1_0: the per-block partial sums, added by a second kernel), eager and in
    a CUDA graph with dependent launch: the graph's outputs equal the eager
    ones bit for bit, and the eager ones match the oracle on sampled rows."""
    M, T = 8, 3
    c = synth.make_case(wl, M=M)
    n, k = c.values.shape
    pay = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    s = dev_signs(c.signs)
    xv, xraw = synth.activations(np.random.default_rng(31), T * M, k, "bf16")
    xs = [torch.from_numpy(np.ascontiguousarray(xraw[M * t:M * (t + 1)]).view(np.int16)).to(DEV).view(torch.bfloat16)
          for t in range(T)]
    need = nt.ninfer_ternary_matmul_workspace(fmt, n, k, M, True)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)

    def calls(ys):
        for t in range(T):
            nt.ninfer_ternary_matmul(fmt, pay, n, k, xs[t], s, y=ys[t], workspace=ws)

    y_e = [torch.empty((M, n), dtype=torch.float32, device=DEV) for _ in range(T)]
    calls(y_e)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(9).integers(0, n, 1000)]))
    ref = oracle.ternary_matmul(fmt, oracle.pack_planes(fmt, c.values[rows], c.scales[rows]), rows.size, k, xv,
                                signs_values(c))
    got = np.concatenate([y.cpu().numpy() for y in y_e])[:, rows].astype(np.float64)
    check_decode(got, ref)
    y_g = [torch.full((M, n), float("nan"), dtype=torch.float32, device=DEV) for _ in range(T)]
    g = _graph(lambda: calls(y_g))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(y_g[t], y_e[t]), t
    assert nt.ninfer_device_errors() == 0


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_prefill_graph_replay_shared_workspace(fmt):
    """Prefill (M = 300 on a 1100 x 2048 matrix), two calls back to back through
    one shared workspace (the rotated binary16 activations; for PTQ1_0 also the
    planes rewritten as PQ2_0), eager and in a CUDA graph: the graph's outputs
    equal the eager ones bit for bit, and the eager ones match the oracle on
    every output."""
    M, T = 300, 2
    c = synth.make_case("prefill", n=1100, k=2048, M=M, seed=12)
    n, k = c.values.shape
    pay = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    s = dev_signs(c.signs)
    xv, xraw = synth.activations(np.random.default_rng(41), T * M, k, "bf16")
    xs = [torch.from_numpy(np.ascontiguousarray(xraw[M * t:M * (t + 1)]).view(np.int16)).to(DEV).view(torch.bfloat16)
          for t in range(T)]
    need = nt.ninfer_ternary_matmul_workspace(fmt, n, k, M, True)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)

    def calls(ys):
        for t in range(T):
            nt.ninfer_ternary_matmul(fmt, pay, n, k, xs[t], s, y=ys[t], workspace=ws)

    y_e = [torch.empty((M, n), dtype=torch.float32, device=DEV) for _ in range(T)]
    calls(y_e)
    torch.cuda.synchronize()
    ref = oracle.ternary_matmul(fmt, oracle.pack_planes(fmt, c.values, c.scales), n, k, xv, signs_values(c))
    check_prefill(np.concatenate([y.cpu().numpy() for y in y_e]).astype(np.float64), ref)
    y_g = [torch.full((M, n), float("nan"), dtype=torch.float32, device=DEV) for _ in range(T)]
    g = _graph(lambda: calls(y_g))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(y_g[t], y_e[t]), t
    assert nt.ninfer_device_errors() == 0


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_embed_graph_replay(fmt):
    """Three embedding gathers (16 ids each, repeats included) back to back,
    eager and in a CUDA graph: equal bit for bit; the eager rows match the
    oracle."""
    c = synth.make_case("gateup", n=2000, k=5120, M=1, seed=23)
    n, k = c.values.shape
    pay = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
    s = dev_signs(c.signs)
    T = 3
    ids_np = np.random.default_rng(24).integers(0, n, (T, 16)).astype(np.int32)
    ids_np[1, 3] = ids_np[1, 4]
    ids = [torch.from_numpy(ids_np[t].copy()).to(DEV) for t in range(T)]

    def calls(outs):
        for t in range(T):
            nt.ninfer_ternary_embed(fmt, pay, n, k, ids[t], s, out=outs[t])

    o_e = [torch.empty((16, k), dtype=torch.float32, device=DEV) for _ in range(T)]
    calls(o_e)
    torch.cuda.synchronize()
    ref = oracle.embed_rows(fmt, oracle.pack_planes(fmt, c.values, c.scales), n, k, ids_np.reshape(-1), signs_values(c))
    check_decode(np.concatenate([o.cpu().numpy() for o in o_e]).astype(np.float64), ref)
    o_g = [torch.full((16, k), float("nan"), dtype=torch.float32, device=DEV) for _ in range(T)]
    g = _graph(lambda: calls(o_g))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(o_g[t], o_e[t]), t
    assert nt.ninfer_device_errors() == 0


def _sweep_shapes():
    """24 seeded decode shapes per format: n in [1, 1500], k a multiple of 1024
    up to 12288 (the rotated path), M in {1, 2, ..., 8}; they cover single CTAs,
    ragged last CTAs, clusters of two and four and both M = 1 kernels' fallbacks."""
    rng = np.random.default_rng(2026)
    out = []
    for fmt in ("PQ2_0_G128", "PTQ1_0_G128"):
        for i in range(24):
            n = int(rng.integers(1, 1501))
            k = 1024 * int(rng.integers(1, 13))
            M = 1 if i % 2 == 0 else int(rng.integers(2, 9))
            out.append((fmt, n, k, M))
    return out


@pytest.mark.parametrize("fmt,n,k,M", _sweep_shapes())
def test_matmul_decode_shape_sweep(fmt, n, k, M):
    c = synth.make_case("gateup", n=n, k=k, M=M, seed=1000 + n + k + M)
    y = run_matmul(fmt, c)
    ref = oracle_matmul_rows(fmt, c, np.arange(n))
    check_decode(y, ref)


def _prefill_sweep_shapes():
    """8 seeded prefill shapes per format: M in [9, 700] (ragged 192-token
    tiles), n in [1, 1500] (ragged 128-row tiles), k a multiple of 1024 up to 4096."""
    rng = np.random.default_rng(2027)
    return [(fmt, int(rng.integers(1, 1501)), 1024 * int(rng.integers(1, 5)), int(rng.integers(9, 701)))
            for fmt in ("PQ2_0_G128", "PTQ1_0_G128") for _ in range(8)]


@pytest.mark.parametrize("fmt,n,k,M", _prefill_sweep_shapes())
def test_matmul_prefill_shape_sweep(fmt, n, k, M):
    c = synth.make_case("prefill", n=n, k=k, M=M, seed=2000 + n + k + M)
    y = run_matmul(fmt, c)
    ref = oracle_matmul_rows(fmt, c, np.arange(n))
    check_prefill(y, ref)
