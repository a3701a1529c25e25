"""Plain fp64 CPU oracle for the batched prefill of one Gated DeltaNet layer.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import anything from this package.  The CUDA
library never calls it, and it shares no code with the CUDA library: the two
sides meet only through the seeded inputs of
``hybrid_gated_deltanet_q4k_gb300.synth``.

What it computes follows the pages on the subject (issue and pull-request
threads on Qwen3.5 prefill speed):

* ``q4k``    the GGUF Q4_K superblock (256 values, 8 sub-blocks of 32, 6-bit
  scales and mins, fp16 d/dmin), its decode to exact fp32, and a plain
  min-max encoder;
* ``q6k``    the GGUF Q6_K superblock (256 values, 16 sub-blocks of 16, int8
  scales, fp16 d, 6-bit codes split into 4 + 2 bits), its exact decode and a
  plain absmax encoder;
* ``quant``  int8 row quantisation with one fp32 scale per row, the exact
  integer product of two int8 matrices and its fp32 rescale, bf16 rounding;
* ``attention``  causal grouped-query softmax attention (the prefill of the
  hybrid model's full-attention layers), in float64;
* ``layer``  the causal 4-tap conv with SiLU, per-head L2 norm, the gates,
  the gated delta rule one token at a time (and, to pin the algebra a chunked
  kernel uses, its chunked WY/UT form), the gated RMSNorm and the whole layer.

Encodings (Q4_K, int8, the integer product and its fp32 rescale, bf16
rounding) are emulated bit for bit in numpy float32/int; everything else runs
in float64, with the recurrence one token at a time.

Every function carries its own pins in ``tests/test_oracle_*.py`` (closed
forms, invariants, brute force on tiny inputs).  The whole-layer composition
has no worked example on the pages, so its end-to-end values are pinned only
through the pinned stages and the layer-level invariants (extend equals
re-prefill, chunked equals sequential).
"""
from . import q4k, q6k, quant, layer, attention  # noqa: F401
