"""CPU oracle of the routed MoE-FFN step (float64).

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg may use it; the library never does.
"""
