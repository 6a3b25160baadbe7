"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only *draws* inputs (random numbers, shapes, positions, poison
rows, the rotary embedding's cos/sin tables).  It holds none of the attention
or rotation arithmetic, so both the CUDA path and the CPU oracle can consume
its outputs without sharing any of the method's code.
"""

from .generators import (  # noqa: F401
    DecodeCase,
    PrefillCase,
    decode_case,
    prefill_case,
    streaming_inputs,
    rope_tables,
    bf16_from_f32,
    WORKLOADS,
)
