"""CPU oracle for the fused MoE layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 NumPy restatement of what the layer computes, used to check
the CUDA path.  Only the test suite, the smoke check and the benchmark's CPU
baseline leg may import it; the library itself never does, and the oracle
never imports the library (they share only the seeded input recipe in
``mixture_experts_layer_19_gb300.workload``).

Modules:
  moe_ref -- routing, layout, SwiGLU experts, combine, backward (BF16,
             MXFP8 and NVFP4 quantisation points), router GEMM.
  mxfp8   -- OCP MX v1.0 E8M0 block scale + OCP FP8 E4M3 element codec.
  nvfp4   -- E2M1 elements, E4M3 scale per 16 elements, fp32 tensor scale.

Parity pins for every function live in ``tests/test_oracle_*.py``; no oracle
function is unpinned.
"""
