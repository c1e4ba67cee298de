"""The oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_oracle_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.row_split_geometry("Q4_0", 4, 128)
    with pytest.raises(ValueError):
        oracle.row_split_geometry("PQ2_0_G128", 0, 128)
    with pytest.raises(ValueError):
        oracle.hadamard_forward(np.ones((1, 1000)), np.ones(1000))
    with pytest.raises(ValueError):
        oracle.hadamard_forward(np.ones((1, 1024)), np.full(1024, 0.5))
    with pytest.raises(ValueError):
        oracle.pack_planes("PQ2_0_G128", np.full((1, 128), 2, np.int8), np.zeros((1, 1), np.uint16))
    p = np.zeros(oracle.row_split_geometry("PQ2_0_G128", 1, 128).payload_bytes, np.uint8)
    p[:32] = 0xFF
    with pytest.raises(ValueError):
        oracle.unpack_planes("PQ2_0_G128", 1, 128, p)
    with pytest.raises(ValueError):
        oracle.dequantize("PQ2_0_G128", p[:-1], 1, 128)


def test_padding_encodes_zero():
    """k not a multiple of 128: pad weights are value 0 and never reach y."""
    rng = np.random.default_rng(2)
    for fmt in ("PQ2_0_G128", "PTQ1_0_G128"):
        n, k = 7, 300
        v = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
        s = np.full((n, 3), 0x3C00, np.uint16)
        payload = oracle.pack_planes(fmt, v, s)
        g = oracle.row_split_geometry(fmt, n, k)
        full = oracle.unpack_planes(fmt, n, g.k_pad, _repad(fmt, payload, n, k, g.k_pad))[0]
        assert np.all(full[:, k:] == 0) and np.array_equal(full[:, :k], v)
        x = rng.standard_normal((1, k))
        assert np.allclose(oracle.ternary_matmul(fmt, payload, n, k, x), x @ v.T.astype(np.float64))


def _repad(fmt, payload, n, k, kp):
    # same bytes describe the (n, k_pad) matrix because geometry only uses k_pad
    assert oracle.row_split_geometry(fmt, n, k).payload_bytes == oracle.row_split_geometry(fmt, n, kp).payload_bytes
    return payload
