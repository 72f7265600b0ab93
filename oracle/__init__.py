"""CPU oracle for batch-1 Llama decode.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding) never calls it and has no CPU fallback.

What it computes is the plain definition of a Llama-style dense decoder
(RMSNorm, rotate-half RoPE, grouped-query attention over a bf16 KV cache,
SwiGLU FFN, final norm, untied LM head, greedy argmax), which the persistent
megakernel pages reach by fusion only (AutoMegaKernel explainer, "Methodology":
the megakernel must match HuggingFace greedy decode token for token; Kog
monokernel tutorial: the whole decode loop, LM head sampling included, in one
kernel).  Arithmetic is float64 unless a step fixes a storage precision (the
bf16 KV cache, fp16 quantisation scales).  It shares no code with the GPU path.

Parity pins (tests/test_oracle_*.py): closed forms for RMSNorm, RoPE and
softmax; single-position attention returning V; GQA equal to MHA on repeated
heads; incremental KV-cache decode equal to full causal recompute; brute force
on tiny quantiser rows; the schedule simulator against hand-built schedules
whose safety is known by inspection.
"""
from . import llama, quant, sampling, schedule_sim  # noqa: F401
