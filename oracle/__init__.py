"""fp64 CPU oracle for the Beam MoE sublayer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the sublayer computes,
written from three public pages about serving Reflection Beam 501B-A23B:

* the TokenSpeed blog on Reflection Beam (lightseek.org), sections
  "Model architecture and precision -> Architecture", "Fused FP32 routing",
  "MNNVL all-reduce and SandwichNorm fusion" and "TensorRT-LLM NVFP4 MoE";
* the Gaudi cookbook port "Beam-1.0-501B-A23B on Gaudi 2", section
  "What was built -> Model code" (fp32 router, bf16 rounding points);
* the vLLM Beam summary (agentlenshq), section "MoE and residual stream:
  FP32 router, sandwich norm, depth-scaled residual" and change 1 of the
  seven kernel changes (norm / residual / norm fusion).

Everything is computed in float64; bf16 values are exact in float64 and the
only roundings are the bf16 rounding points the pages name. The oracle shares
no code with the CUDA library and never imports it. Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may use
this package; the product path must never route through it.

Pins (what checks the oracle against something other than itself) live in
``tests/test_oracle_*.py``. Parity unpinned: agreement with the real Beam
model, whose code and weights are not available (group-score rule and the
exact placement of rounding inside the norm follow the plainest reading).
"""
from . import bf16, boundary, routing, permute, experts, combine, layer  # noqa: F401
