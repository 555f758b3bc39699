"""Seeded synthetic inputs for fused linear cross-entropy.

This package is shared by the oracle tests, the GPU parity tests and the
benchmark.  It draws random numbers, rounds them to bf16 and builds the target,
ignore-mask and upstream-gradient recipes of each workload.  It holds none of
the method's arithmetic (no logits, no softmax, no gradient).
"""

from .synth import (  # noqa: F401
    IGNORE_INDEX,
    WORKLOADS,
    Inputs,
    Workload,
    bf16_bits_from_f32,
    bf16_bits_to_f32,
    bf16_bits_to_f64,
    generate,
    inputs_digest,
    workload,
)
