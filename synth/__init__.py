"""Seeded synthetic inputs for the ternary projection workloads.

This module only draws random numbers and rounds them to the storage types the
inputs have (binary16 group scales, bfloat16 sign vectors and activations).
It holds no step of the method itself: no packing, no decoding, no transform
and no contraction. Both the CUDA path's tests/benchmark and the CPU oracle's
callers take their inputs from here, so the two sides see identical inputs
while sharing no code that computes anything.

Distributions (the workload recipe):
  * ternary values iid from {-1, 0, +1} with probabilities (0.3, 0.4, 0.3);
  * one binary16 scale per 128-weight group, U[0.005, 0.05] rounded to nearest;
  * sign vector D iid +-1 stored as bfloat16;
  * activations N(0, 1), stored as bfloat16 (float32 for the tiny case);
  * token ids uniform in [0, vocab).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GROUP = 128          # weights per scale group (both ternary formats)
HADAMARD_BLOCK = 1024

FORMAT_IDS = {"PQ2_0_G128": 142, "PTQ1_0_G128": 143}


# ----------------------------------------------------------------------------
# storage-type rounding (input preparation only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    rounding_bias = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding_bias) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 values (exact)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def f16_bits(a) -> np.ndarray:
    """Round to IEEE binary16 (numpy's nearest-even cast); return uint16 bits."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------
# individual generators
# ----------------------------------------------------------------------------
def ternary_values(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """n x k int8 values in {-1, 0, +1} with P = (0.3, 0.4, 0.3)."""
    u = rng.integers(0, 10, size=(n, k), dtype=np.uint8)
    v = np.zeros((n, k), dtype=np.int8)
    v[u < 3] = -1
    v[u >= 7] = 1
    return v


def group_scales(rng: np.random.Generator, n: int, groups: int) -> np.ndarray:
    """n x groups binary16 bit patterns of U[0.005, 0.05]."""
    return f16_bits(rng.uniform(0.005, 0.05, size=(n, groups)))


def sign_vector(rng: np.random.Generator, K: int) -> np.ndarray:
    """K bfloat16 bit patterns of iid +-1 (0x3F80 = +1, 0xBF80 = -1)."""
    neg = rng.integers(0, 2, size=K, dtype=np.uint8).astype(bool)
    return np.where(neg, np.uint16(0xBF80), np.uint16(0x3F80)).astype(np.uint16)


def activations(rng: np.random.Generator, M: int, k: int, dtype: str):
    """M x k activations N(0,1). Returns (float32 values, raw storage array).

    dtype 'bf16': raw is uint16 bfloat16 bits and the values are their exact
    float32 widening. dtype 'f32': raw is the float32 array itself.
    """
    x = rng.standard_normal(size=(M, k)).astype(np.float32)
    if dtype == "bf16":
        raw = f32_to_bf16_bits(x)
        return bf16_bits_to_f32(raw), raw
    if dtype == "f32":
        return x, x
    raise ValueError(f"unknown activation dtype {dtype!r}")


def token_ids(rng: np.random.Generator, count: int, vocab: int) -> np.ndarray:
    return rng.integers(0, vocab, size=count, dtype=np.int64).astype(np.int32)


# ----------------------------------------------------------------------------
# workload presets
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str
    n: int
    k: int
    M: int
    x_dtype: str
    seed: int
    rotate: bool = True
    description: str = ""
    mats: int = 1            # 2: FFN gate and up projections of one activation (SwiGLU product)
    kind: str = "matmul"     # "embed": gather EMBED_COUNT rows and inverse-rotate them


WORKLOADS = {
    "tiny": Workload("tiny", "PQ2_0_G128", 256, 1024, 1, "f32", 0,
                     description="PQ2_0_G128 matvec n=256 k=1024 (one Hadamard block), M=1, fp32 x"),
    "gateup": Workload("gateup", "PQ2_0_G128", 17408, 5120, 1, "bf16", 1,
                       description="FFN gate/up decode GEMV, PQ2_0_G128 n=17408 k=5120 (5 Hadamard blocks), M=1"),
    "down": Workload("down", "PTQ1_0_G128", 5120, 17408, 1, "bf16", 2,
                     description="FFN down decode GEMV, PTQ1_0_G128 n=5120 k=17408 (17 Hadamard blocks), M=1"),
    "down_m8": Workload("down_m8", "PTQ1_0_G128", 5120, 17408, 8, "bf16", 2,
                        description="FFN down decode GEMV, PTQ1_0_G128 n=5120 k=17408, M=8"),
    "prefill": Workload("prefill", "PQ2_0_G128", 17408, 5120, 2048, "bf16", 3,
                        description="prefill GEMM, PQ2_0_G128 n=17408 k=5120, M=2048 token rows"),
    "prefill_down": Workload("prefill_down", "PTQ1_0_G128", 5120, 17408, 2048, "bf16", 5,
                             description="prefill GEMM, PTQ1_0_G128 n=5120 k=17408 (FFN down), M=2048 token rows"),
    "ffn_gate_up": Workload("ffn_gate_up", "PQ2_0_G128", 17408, 5120, 1, "bf16", 6,
                            description="FFN gate and up projections, PQ2_0_G128 17408x5120 each with its own "
                                        "sign vector, SwiGLU product, M=1", mats=2),
    "embed": Workload("embed", "PQ2_0_G128", 248320, 5120, 1, "bf16", 4,
                      description="embedding: 64 token ids uniform in [0, 248320) gathered from the PQ2_0_G128 "
                                  "head matrix 248320x5120, dequantised, inverse transform D*(H*e)/32",
                      kind="embed"),
    "head": Workload("head", "PQ2_0_G128", 248320, 5120, 1, "bf16", 4,
                     description="output head, PQ2_0_G128 n=248320 k=5120, M=1"),
    "head_m8": Workload("head_m8", "PQ2_0_G128", 248320, 5120, 8, "bf16", 4,
                        description="output head, PQ2_0_G128 n=248320 k=5120, M=8"),
    "head_ptq1": Workload("head_ptq1", "PTQ1_0_G128", 248320, 5120, 1, "bf16", 4,
                          description="output head, PTQ1_0_G128 n=248320 k=5120 (278,118,400-byte payload), M=1"),
    "head_ptq1_m8": Workload("head_ptq1_m8", "PTQ1_0_G128", 248320, 5120, 8, "bf16", 4,
                             description="output head, PTQ1_0_G128 n=248320 k=5120, M=8"),
    "embed_ptq1": Workload("embed_ptq1", "PTQ1_0_G128", 248320, 5120, 1, "bf16", 4,
                           description="embedding: 64 token ids uniform in [0, 248320) gathered from the PTQ1_0_G128 "
                                       "head matrix 248320x5120, dequantised, inverse transform D*(H*e)/32",
                           kind="embed"),
}

EMBED_COUNT = 64     # gathered embedding rows for the embedding workload (seed 4, head matrix)


@dataclass
class Case:
    """All inputs of one workload, in storage form."""
    workload: Workload
    values: np.ndarray       # n x k int8 ternary values
    scales: np.ndarray       # n x groups uint16 (binary16 bits)
    signs: np.ndarray        # k uint16 (bfloat16 bits), or empty when not rotated
    x: np.ndarray            # M x k float32 values (exactly representable in x_dtype)
    x_raw: np.ndarray        # M x k storage array (uint16 bf16 bits or float32)
    ids: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    up: tuple | None = None  # (values, scales, signs) of the up projection when workload.mats == 2


def up_projection(seed: int, n: int, k: int):
    """The second projection of a gate/up pair: values, scales and signs drawn
    in that order from default_rng(seed), with the distributions above."""
    rng = np.random.default_rng(seed)
    return ternary_values(rng, n, k), group_scales(rng, n, -(-k // GROUP)), sign_vector(rng, k)


def make_case(w: Workload | str, n: int | None = None, k: int | None = None,
              M: int | None = None, seed: int | None = None, with_ids: bool = False) -> Case:
    """Draw every input of a workload in a fixed order from default_rng(seed).

    Order: values, scales, signs, activations, ids. n/k/M/seed override the
    preset (smaller shapes with the same distributions for parity tests). A
    two-projection workload also draws the up projection from up_projection(seed + 1000).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = w.n if n is None else n
    k = w.k if k is None else k
    M = w.M if M is None else M
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    groups = -(-k // GROUP)
    values = ternary_values(rng, n, k)
    scales = group_scales(rng, n, groups)
    signs = sign_vector(rng, k) if w.rotate else np.zeros(0, np.uint16)
    x, x_raw = activations(rng, M, k, w.x_dtype)
    ids = token_ids(rng, EMBED_COUNT, n) if with_ids else np.zeros(0, np.int32)
    up = up_projection(seed + 1000, n, k) if w.mats == 2 else None
    return Case(w, values, scales, signs, x, x_raw, ids, up)
