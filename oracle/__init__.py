"""Plain f64 CPU oracle of the quantized GEMV and the routed-expert MLP.

Test infrastructure: only the tests, the package entry's smoke check and the
bench's CPU-baseline leg use it; the CUDA library never does.
"""
