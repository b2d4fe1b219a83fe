"""CPU oracle for the fused MoE layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 NumPy restatement of what the layer computes, used to check
the CUDA path.  Only the test suite, the smoke check and the benchmark's CPU
baseline leg may import it; the library itself never does, and the oracle
never imports the library (they share only the seeded input recipe in
``mixture_experts_layer_19_gb300.workload``).

Modules:
  moe_ref -- routing, layout, SwiGLU experts, combine, backward (BF16 and
             MXFP8 quantisation points).
  mxfp8   -- OCP MX v1.0 E8M0 block scale + OCP FP8 E4M3 element codec.

Parity pins for every function live in ``tests/test_oracle_*.py``; no oracle
function is unpinned.
"""
