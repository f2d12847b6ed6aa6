"""CPU oracle for gated GQA attention -- test infrastructure only.

Only tests/, the package smoke check and the benchmark's CPU-baseline leg may import
this package. The product path never does: it runs the CUDA kernels or fails.
"""
