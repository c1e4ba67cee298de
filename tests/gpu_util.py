"""Helpers for the GPU parity tests: inputs from synth, payloads packed by the
library's host packer, device copies, and oracle references computed from the
same generator output (never from anything the CUDA path produced)."""
import numpy as np
import torch

import bit_gemv_gb300 as nt
import oracle
import synth

DEV = torch.device("cuda:0")


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def dev_signs(signs_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(signs_bits).view(np.int16)).to(DEV)


def dev_x(case) -> torch.Tensor:
    if case.workload.x_dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(case.x_raw).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(case.x)).to(DEV)


def signs_values(case) -> np.ndarray:
    return synth.bf16_bits_to_f32(case.signs).astype(np.float64)


def oracle_matmul_rows(fmt, case, rows, rotate=True):
    """Oracle y for a subset of rows: the oracle packs exactly those rows of the
    generator's values/scales itself, then decodes and contracts."""
    rows = np.asarray(rows)
    sub = oracle.pack_planes(fmt, case.values[rows], case.scales[rows])
    return oracle.ternary_matmul(fmt, sub, rows.size, case.values.shape[1], case.x,
                                 signs_values(case) if rotate else None)


def run_matmul(fmt, case, rotate=True, y_dtype=torch.float32, payload_dev=None):
    n, k = case.values.shape
    if payload_dev is None:
        payload_dev = dev_u8(nt.ninfer_ternary_pack(fmt, case.values, case.scales))
    y = nt.ninfer_ternary_matmul(fmt, payload_dev, n, k, dev_x(case),
                                 dev_signs(case.signs) if rotate else None, y_dtype=y_dtype)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)
