"""Seeded synthetic inputs for CSR-indexed sparse and paged attention.

This module is shared by the oracle tests, the GPU parity tests and the benchmark.
It holds no attention, rotary or quantisation arithmetic: only seeded random draws,
index structures (CSR block masks, page tables, sparse row lists) and dtype casts
done by torch. The rotary cos/sin cache is an input of the method, so it is built
here as well (float64 formula, stored as float32), and both sides read the same
stored values.
"""

from .gen import (  # noqa: F401
    bsr_inputs,
    variable_block_inputs,
    paged_decode_inputs,
    paged_prefill_inputs,
    mla_inputs,
    mla_paged_inputs,
    mla_append_inputs,
    E4M3_NAN,
    rope_cos_sin_cache,
    CONFIGS,
    make,
)
