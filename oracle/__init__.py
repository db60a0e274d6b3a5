"""CPU oracle for the single-GPU MoE layer hot path (route, permute, experts, combine).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import anything here.
The product path (the CUDA library and its Python binding) never imports, calls or
links this package, and this package shares no code with it: no kernels, headers,
helpers, tables or constant generators.  The only module both sides use is the seeded
input generator ``combine_moe_route_softmax_gb300.synth``, which holds none of the
method's arithmetic.

Plain, slow, obviously correct numpy.  Every function cites the passage of the source
pages it follows; the pages are four pull-request pages:

* "Add MoE dispatch/combine fake quantization for vLLM's DeepGEMM Mega-MoE"
  (NVIDIA Model-Optimizer PR #2767) -- the combine contract.
* "[Kernel] DeepEP dispatch-combine kernel integration" (vLLM PR #18434) -- FP8
  dispatch with scales, block tile counts, router-weight placement.
* "[Distributed][MoonEP] BF16 integration of MoonEP balanced EP backend" (vLLM PR
  #52101) -- the expert-major layout ([NvS, H] rows plus cu_seqlens), the grouped
  gate/up/down experts and the dense per-token reference MoE.
* "[Bugfix][MoE] Size the permute scratch from its inputs" (vLLM PR #60447) -- scratch
  sized from the inputs, padding buckets.

Precision: floating point is fp64 except where the pages fix it.  The combine's
precision is fixed by the Mega-MoE page (FP32 from zero, one BF16 rounding), so the
combine is written in explicit float32 steps; the FP8 quantisers take their rounding
decision in float32, the precision the kernel computes in.

Parity pins: every function here is checked in ``tests/test_oracle_*.py`` against
brute force, closed forms, invariants or library routines.  None is "parity unpinned".
"""
