"""fp64 CPU oracle of the SparDA forecast-driven block-sparse decode step.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The CUDA product path never imports it.
"""
