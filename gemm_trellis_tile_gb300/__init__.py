"""Trellis-coded (EXL3-style, cb=1) linear layers on one sm_103a GPU.

The compute lives in libescha.so (CUDA, C ABI in include/escha.h); `escha`
is its Python binding, `synthetic` the seeded input generator and `workloads`
the byte/flop accounting used by the benchmark.
"""
