"""Routed Mixture-of-Experts SwiGLU FFN forward pass for GB300 (sm_103a).

The compute lives in ``libmoeffn.so`` (hand-written CUDA, C ABI declared in
``include/moe_ffn.h``); ``moe_ffn`` is its thin ctypes binding.  ``synth``
holds the seeded synthetic-input recipe and the workload table.
"""
