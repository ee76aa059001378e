"""CPU oracle for document-masked context-parallel attention.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package. The library path never
calls it; it shares no code with the CUDA kernels or the C++ planner.

Modules:
  attention  fp64 forward, backward and (O, LSE) merge, written from their
             plain definitions (numpy).
  plan       the sharding policies (Llama3 2xCP, Per-Doc, Whole-Doc, hybrid
             Algorithm 1), the workload model and the communication volumes.
"""
