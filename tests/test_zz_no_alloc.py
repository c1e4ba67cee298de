"""The allocation-free projection entry point (GPU).

ninfer_ternary_matmul_noalloc serves callers that cannot allocate device
memory (for example a plug-in that only receives its input and output
buffers): it takes its workspace from a fixed array inside the library
instead of from the caller. This file checks, through the C ABI, that it
returns what ninfer_ternary_matmul returns with a caller-allocated workspace,
on two calls in a row sharing that array, and that it refuses problems larger
than the array. It sits in its own file, collected last, so that a run that
stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_gemv_gb300 as nt
import synth
from gpu_util import DEV, dev_signs, dev_u8, dev_x

pytestmark = pytest.mark.gpu

TOL = {True: 1e-3, False: 2e-2}     # decode (M <= 8) / prefill: the parity tests' infinity-norm bounds


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _noalloc(fmt_id, payload, n, k, x, signs, y):
    """One call of the new entry point straight through the C ABI (ctypes)."""
    lib = ctypes.CDLL(nt.LIBRARY_PATH)
    fn = lib.ninfer_ternary_matmul_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_uint64, ctypes.c_void_p]
    x_dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[x.dtype]
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return fn(fmt_id, payload.data_ptr(), payload.numel(), n, k, x.data_ptr(), x_dt,
              signs.data_ptr() if signs is not None else None, y.data_ptr(), 0, x.shape[0], stream)


# Every case is one whose path takes a workspace, so the built-in array is
# written and read: per-block partial sums (PTQ1_0, 2 <= M <= 8), binary16
# activation fragments (PQ2_0, 2 <= M <= 8), and on the prefill path the
# rotated binary16 activations (PQ2_0) plus the PTQ1_0 planes rewritten as
# PQ2_0 planes.
@pytest.mark.parametrize("fmt,n,k,M", [("PTQ1_0_G128", 300, 2048, 3), ("PQ2_0_G128", 517, 5120, 4),
                                       ("PQ2_0_G128", 200, 2048, 24), ("PTQ1_0_G128", 64, 1024, 16)])
def test_noalloc_matches_workspace_entry_two_calls(fmt, n, k, M):
    fmt_id = nt.FORMATS[fmt]
    need = nt.ninfer_ternary_matmul_workspace(fmt, n, k, M, True)
    assert 0 < need <= nt.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((31, 32)):          # two calls in a row share the scratch array
        c = synth.make_case("gateup", n=n, k=k, M=M, seed=seed)
        payload = dev_u8(nt.ninfer_ternary_pack(fmt, c.values, c.scales))
        x, signs = dev_x(c), dev_signs(c.signs)
        ref = nt.ninfer_ternary_matmul(fmt, payload, n, k, x, signs)
        y = torch.full((M, n), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(fmt_id, payload, n, k, x, signs, y) == 0, nt._lib.ninfer_last_error()
        torch.cuda.synchronize()
        got, want = y.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert _rel(got, want) <= TOL[M <= 8], f"call {call}: rel {_rel(got, want)}"


def test_noalloc_rejects_problem_larger_than_scratch():
    fmt, n, k, M = "PTQ1_0_G128", 64, 17408, 128
    need = nt.ninfer_ternary_matmul_workspace(fmt, n, k, M, True)
    assert need > nt.NOALLOC_SCRATCH_BYTES
    g = nt.ninfer_ternary_geometry(fmt, n, k)
    payload = torch.zeros(g.payload_bytes, dtype=torch.uint8, device=DEV)
    x = torch.zeros((M, k), dtype=torch.bfloat16, device=DEV)
    signs = torch.zeros(k, dtype=torch.int16, device=DEV)
    y = torch.zeros((M, n), dtype=torch.float32, device=DEV)
    st = _noalloc(nt.FORMATS[fmt], payload, n, k, x, signs, y)
    assert st == 4                                   # NINFER_ERR_SIZE_MISMATCH, nothing launched
    assert b"scratch" in nt._lib.ninfer_last_error()
