"""Plain float64 CPU oracle for CSR-indexed sparse and paged attention.

TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the CPU
baseline leg of the benchmark may import this package; the product path never does.
It shares no code with the CUDA library: it decodes stored bf16/fp16/E4M3 bits
itself, applies the rotary embedding itself, and computes attention as the plain
dense definition (masked softmax) with numpy.

Sources (web pages describing the method; cited by title and section):
  * "flashinfer.sparse - FlashInfer 0.7.4 documentation": BlockSparseAttentionWrapper
    (class description, the 3x3 worked example, plan() and run() parameters).
  * "Sparse MLA" (MATE 0.2.6 API docs): mla_rope_quantize_fp8 and sparse_mla_fp8_decode.
  * "FlashInfer Compatibility Wrapper" (MATE 0.2.6 docs): RoPE and FP8 quantization,
    Sparse MLA decode, scale folding.
  * "FlashInfer" agent-skill summary: KV-Cache Formats (paged KV-cache), Cascade Inference.
  * FlashInfer cheat page: docs/api/cascade.rst (merge_state / merge_states).

Parity pins: every function here is pinned by the not-gpu tests in tests/ against
values fixed by the pages or by mathematics (worked example, library routines on
special cases, closed forms, invariants, brute force). The plan restatement in
plan_ref.py is pinned by invariants (every unit and token covered exactly once,
balance bounds) rather than by a value printed on the pages, which give no
partition rule.
"""

from . import numerics, rope, attention, plan_ref  # noqa: F401
