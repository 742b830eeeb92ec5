"""Split-KV exact attention for long-context decode, and fused causal prefill, on B300.

The compute path is the CUDA library ``libta.so`` (C ABI in include/ta.h);
``ta`` is its Python binding.  ``synth`` holds the seeded workload inputs and
``accounting`` the byte/FLOP counts used for roofline figures.
"""
