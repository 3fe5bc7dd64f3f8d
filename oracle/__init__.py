"""fp64 CPU oracles for the fused, chunked top-K KL loss.

TEST INFRASTRUCTURE: imported only by the test suite, the package smoke check
and the benchmark's CPU-baseline leg. Nothing on the product path imports it.
"""
