"""CPU oracle for the quantized-linear path.  TEST INFRASTRUCTURE ONLY.

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this package.  The library (`w4a4_precision_gemm_gb300`) never
imports it and has no CPU fallback.  The oracle shares no code with the CUDA
path: the two meet only through the seeded input generator in `synth`.

The oracle is plain numpy, written to be checked against the pages by eye:

* `codecs`  - E4M3FN, E5M2, E2M1, E8M0 and INT8 codes, defined from the bit
  layouts ("Low-bit LLM Weights and Activations", section 2.2 table "FP8 Format
  Comparison (OCP OFP8 1.0)" and section 2.4 "FP4 / NVFP4"); encoding is
  round-to-nearest-even onto the decoded grid, saturating at the largest
  finite value.
* `quant`   - the dynamic quantizers: FP8 per token / per 1x128 group / per
  128x128 weight block, INT8 with optional SmoothQuant factors, NVFP4 and MXFP4
  ("FP8 and FP4 inference, SmoothQuant and activation quantization", sections
  "Scale granularity" and "Implementation sketch"; "FP8 and INT8 Inference",
  section 5 "INT8 in practice").
* `smooth`  - SmoothQuant calibration ("Low-bit LLM Weights and Activations",
  section 4.2).
* `gemm`    - the dequantized product in fp64 and the factored epilogue
  ("FP8 and FP4 inference ...", section "Scale granularity"; "Low-bit LLM
  Weights and Activations", section 3.4).

Quantizer arithmetic is fp32 because the pages fix it (their emulation runs in
fp32 and names an "fp32 tensor scale"); every `/` is numpy's correctly rounded
fp32 division.  GEMM references are fp64 (exact for products of decoded codes
and fp32 scales) or exact integers for INT8.

Readings of points the pages leave open are listed in each function's
docstring.  Parity of the MXFP4 scale rule is not fixed by the pages (they give
only "power-of-two scale per 32, E8M0, bias 127"); the rule taken is the OCP MX
one: parity unpinned for that choice, checked only through invariants.
"""
