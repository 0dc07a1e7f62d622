"""CPU oracle for trellis-coded linear layers -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import anything under this directory.  The CUDA library never does,
and this package imports nothing from the CUDA library.
"""
