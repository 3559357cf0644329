"""CPU oracle for the quantized KV cache — TEST INFRASTRUCTURE ONLY.

A plain, slow, readable restatement of what the GPU path computes, written in
numpy from the pages' definitions:

* ``oracle.kivi``      KIVI asymmetric 2/4-bit group quantization (keys per
                       channel, values per token, groups of 32 tokens, an fp16
                       residual window that is flushed when it fills), in the
                       IEEE fp32 arithmetic the formula fixes.
* ``oracle.fp8``       FP8 E4M3 encoding from the format definition and the
                       per-tensor dynamic scale ``amax / 448``.
* ``oracle.attention`` single-token decode attention softmax(q K^T / sqrt(d)) V
                       in float64 over exactly the dequantized values.
* ``oracle.layout``    the byte layout of the packed cache, written from its
                       specification in the library header.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The product path (the CUDA library and its Python
binding) never imports, calls or links anything here, and shares no code
with it; the only module both sides read is the seeded input generator
``quantized_kv_cache_quant_gb300.workloads``, which holds no arithmetic of the
method.

Parity pins: every function here is pinned by tests under ``tests/`` (marked
``not gpu``) against closed forms, brute force on tiny inputs, worked numbers
printed on the pages, library routines for special cases, or invariants.
Parity is unpinned only for model quality (perplexity and task accuracy),
which needs trained weights and datasets and is out of scope.
"""
