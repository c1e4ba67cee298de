"""CPU oracle for the Hadamard-rotated ternary projection (TEST INFRASTRUCTURE).

This package is the slow, obviously-correct reference the CUDA path is checked
against. Only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import it; the product library never does, and the two share no code.

Everything is plain numpy in float64 (or exact integer arithmetic for the
codec), written step by step from the source pages:

* "bonsai三元GGUF模型转ninfer模型01" (ninfer ternary artifact format page):
  §2 ternary numeric formats, §3 row-split plane geometry, §4 block <-> plane
  conversion, §6 constants (block size 1024, normalized Sylvester-Walsh-Hadamard,
  explicit signs).
* "GGUF 完整讲解" (GGUF explainer): §4.3 the Q2_0 dequantisation routine, which
  fixes the 2-bit field order and the offset code -> value mapping.
* NInfer "artifact-container.md" (v3 container spec): §6.1 numeric formats,
  §8 the ``hadamard_signs`` auxiliary input.
* "从 TensorSharp 视角解读 Ternary Bonsai 2 27B" (TensorSharp article): §4.2 the
  transform contract H(D.x)/sqrt(block) and its inverse D.(H.x)/sqrt(block),
  §4.4 where the transforms apply (and the dense gated FFN, read as SwiGLU;
  §4.2: fused gate/up weights keep each projection's own transform).

Pins (tests/test_oracle_pins.py) tie each function to something outside the
oracle: the byte counts the format page prints, a library Hadamard matrix,
closed forms, invariants and brute force on tiny inputs.
"""
from .ternary import (  # noqa: F401
    FORMATS,
    GEOMETRY_FIELDS,
    TernaryFormat,
    row_split_geometry,
    pack_planes,
    unpack_planes,
    planes_to_blocks,
    blocks_to_planes,
    dequantize,
    hadamard_matrix,
    hadamard_forward,
    hadamard_inverse,
    ternary_matmul,
    gate_up_swiglu,
    embed_rows,
    max_rel_error,
    significant_rel_error,
)
