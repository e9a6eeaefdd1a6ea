"""fp64 CPU oracle for exact backward-over-backward (BoB) of softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the tests, the smoke check and the CPU-baseline leg of the benchmark do.  It
shares no code with the CUDA path.
"""
