"""Host side of the boundary (CPU only): the library loads and exports every
symbol the header declares, the host geometry/packer/block conversion match
the oracle bit for bit, and argument errors come back as status codes before
any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import bit_gemv_gb300 as nt
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(ninfer_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(nt.LIBRARY_PATH)
    declared = _declared_functions()
    assert len(declared) >= 12
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    assert set(nt.EXPORTED) == set(declared)
    assert nt.ninfer_abi_version() == 1


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
def test_geometry_matches_oracle(fmt):
    rng = np.random.default_rng(1)
    shapes = [(256, 1024), (17408, 5120), (5120, 17408), (248320, 5120), (1, 1), (3, 130), (7, 127)]
    shapes += [(int(rng.integers(1, 300000)), int(rng.integers(1, 40000))) for _ in range(300)]
    for n, k in shapes:
        assert tuple(nt.ninfer_ternary_geometry(fmt, n, k)) == tuple(oracle.row_split_geometry(fmt, n, k)), (n, k)


@pytest.mark.parametrize("fmt", ["PQ2_0_G128", "PTQ1_0_G128"])
@pytest.mark.parametrize("n,k,seed", [(256, 1024, 0), (33, 300, 1), (5, 5120, 2), (64, 17408, 3), (1, 1, 4)])
def test_pack_unpack_bit_exact(fmt, n, k, seed):
    c = synth.make_case("tiny", n=n, k=k, seed=seed)
    p = nt.ninfer_ternary_pack(fmt, c.values, c.scales)
    assert np.array_equal(p, oracle.pack_planes(fmt, c.values, c.scales))
    v, s = nt.ninfer_ternary_unpack(fmt, n, k, p)
    assert np.array_equal(v, c.values) and np.array_equal(s, c.scales)
    b = nt.ninfer_planes_to_blocks(fmt, n, k, p)
    assert np.array_equal(b, oracle.planes_to_blocks(fmt, n, k, p))
    assert np.array_equal(nt.ninfer_blocks_to_planes(fmt, n, k, b), p)


def test_pack_full_gateup_matches_oracle():
    c = synth.make_case("gateup")
    p = nt.ninfer_ternary_pack("PQ2_0_G128", c.values, c.scales)
    assert p.size == 23674880
    assert np.array_equal(p, oracle.pack_planes("PQ2_0_G128", c.values, c.scales))


def test_unpack_rejects_invalid_codes():
    g = nt.ninfer_ternary_geometry("PQ2_0_G128", 2, 128)
    p = np.zeros(g.payload_bytes, np.uint8)
    p[:64] = 0x55
    p[40] = 0x57                                   # field 0 of row 1 byte 8 holds code 3
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_unpack("PQ2_0_G128", 2, 128, p)
    assert e.value.status == 6 and "row 1" in str(e.value)
    t = nt.ninfer_ternary_geometry("PTQ1_0_G128", 1, 128)
    q = np.zeros(t.payload_bytes, np.uint8)
    q[:24] = 243
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_unpack("PTQ1_0_G128", 1, 128, q)
    assert e.value.status == 6
    q[:24] = 121
    q[t.high_offset] = 81
    with pytest.raises(nt.NinferError):
        nt.ninfer_ternary_unpack("PTQ1_0_G128", 1, 128, q)


def test_host_errors():
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_geometry(99, 4, 128)
    assert e.value.status == 2
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_geometry("PQ2_0_G128", 0, 128)
    assert e.value.status == 3
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_geometry("PQ2_0_G128", 2 ** 62, 2 ** 40)
    assert e.value.status == 8
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_ternary_pack("PQ2_0_G128", np.full((2, 128), 2, np.int8), np.zeros((2, 1), np.uint16))
    assert e.value.status == 6
    lib = ctypes.CDLL(nt.LIBRARY_PATH)
    p = np.zeros(100, np.uint8)
    st = lib.ninfer_ternary_unpack(142, ctypes.c_uint64(1), ctypes.c_uint64(128), p.ctypes.data_as(ctypes.c_void_p),
                                   ctypes.c_uint64(100), p.ctypes.data_as(ctypes.c_void_p),
                                   p.ctypes.data_as(ctypes.c_void_p))
    assert st == 4


def test_wait_limit_setting():
    """The wait-bound hook rejects a negative bound and accepts 0 and the default."""
    with pytest.raises(nt.NinferError) as e:
        nt.ninfer_set_wait_limit(-1)
    assert e.value.status == 1
    nt.ninfer_set_wait_limit(0)
    nt.ninfer_set_wait_limit(nt.WAIT_LIMIT_DEFAULT)


def test_device_entry_points_validate_before_launch():
    """Invalid arguments return a status without touching the device (so this
    runs without a GPU). Fake, aligned addresses stand in for device buffers."""
    lib = nt._lib
    fake = ctypes.c_void_p(1 << 20)
    u64 = ctypes.c_uint64
    # K not a multiple of 1024
    assert lib.ninfer_hadamard_fwd(fake, 0, fake, 0, fake, 1, 1000, None) == 3
    # NULL signs
    assert lib.ninfer_hadamard_inv(fake, 0, fake, 0, None, 1, 1024, None) == 1
    # misaligned x
    assert lib.ninfer_hadamard_fwd(ctypes.c_void_p((1 << 20) + 4), 0, fake, 0, fake, 1, 1024, None) == 5
    g = nt.ninfer_ternary_geometry("PQ2_0_G128", 256, 1024)
    # wrong payload size
    assert lib.ninfer_ternary_matmul(142, fake, g.payload_bytes - 1, 256, 1024, fake, 0, fake, fake, 0, 1,
                                     None, 0, None) == 4
    # unknown format
    assert lib.ninfer_ternary_matmul(7, fake, g.payload_bytes, 256, 1024, fake, 0, fake, fake, 0, 1, None, 0, None) == 2
    # rotated input with k % 1024 != 0
    g2 = nt.ninfer_ternary_geometry("PQ2_0_G128", 256, 1000)
    assert lib.ninfer_ternary_matmul(142, fake, g2.payload_bytes, 256, 1000, fake, 0, fake, fake, 0, 1,
                                     None, 0, None) == 3
    # payload not 256-byte aligned
    assert lib.ninfer_ternary_matmul(142, ctypes.c_void_p((1 << 20) + 16), g.payload_bytes, 256, 1024, fake, 0,
                                     fake, fake, 0, 1, None, 0, None) == 5
    # embed with k % 1024 and signs
    assert lib.ninfer_ternary_embed(142, fake, g2.payload_bytes, 256, 1000, fake, 4, fake, fake, 0, None, None) == 3
    # bad output dtype
    assert lib.ninfer_ternary_embed(142, fake, g.payload_bytes, 256, 1024, fake, 4, fake, fake, 2, None, None) == 1
    msg = lib.ninfer_last_error()
    assert msg and b"dtype" in msg
    ws = u64()
    assert lib.ninfer_ternary_matmul_workspace(142, 256, 1024, 0, 1, ctypes.byref(ws)) == 3


def test_gate_up_and_block_conversion_validate_before_launch():
    """The fused gate/up and the device block conversion check their arguments
    before any device work, so these run without a GPU (fake aligned addresses)."""
    lib = nt._lib
    fake = ctypes.c_void_p(1 << 20)
    g = nt.ninfer_ternary_geometry("PQ2_0_G128", 256, 1024)
    pb = g.payload_bytes

    def gate_up(fmt=142, pg=fake, pu=fake, nbytes=pb, n=256, k=1024, sg=fake, su=fake, y_dtype=0, M=1):
        return lib.ninfer_ternary_gate_up(fmt, pg, pu, nbytes, n, k, fake, 0, sg, su, fake, y_dtype, M, None, 0,
                                          None)

    assert gate_up(su=None) == 1                                      # one sign vector without the other
    assert gate_up(y_dtype=2) == 1                                    # f16 output is not offered
    assert gate_up(nbytes=pb - 2) == 4                                # payload size
    assert gate_up(pu=ctypes.c_void_p((1 << 20) + 16)) == 5           # up payload not 256-byte aligned
    assert gate_up(M=0) == 3
    g2 = nt.ninfer_ternary_geometry("PQ2_0_G128", 256, 1000)
    assert gate_up(nbytes=g2.payload_bytes, k=1000) == 3             # rotated input needs whole blocks
    assert gate_up(fmt=9) == 2
    # device block stream <-> planes: sizes and alignment
    blocks = 256 * g.groups_per_row * 34
    assert lib.ninfer_blocks_to_planes_device(142, 256, 1024, fake, blocks - 34, fake, pb, None) == 4
    assert lib.ninfer_blocks_to_planes_device(142, 256, 1024, fake, blocks, fake, pb + 1, None) == 4
    assert lib.ninfer_planes_to_blocks_device(142, 256, 1024, ctypes.c_void_p((1 << 20) + 8), pb, fake, blocks,
                                              None) == 5


def test_validate_signs():
    """Load-time check of a sign vector: exactly +-1 in bfloat16, K % 1024 == 0."""
    import synth

    rng = np.random.default_rng(3)
    s = synth.sign_vector(rng, 2048)
    nt.ninfer_validate_signs(s)                            # valid
    bad = s.copy()
    bad[1500] = 0x3F00                                     # 0.5
    with pytest.raises(nt.NinferError, match="entry 1500"):
        nt.ninfer_validate_signs(bad)
    bad[1500] = 0x0000                                     # +0
    with pytest.raises(nt.NinferError):
        nt.ninfer_validate_signs(bad)
    with pytest.raises(nt.NinferError, match="multiple of 1024"):
        nt.ninfer_validate_signs(s[:1000])
