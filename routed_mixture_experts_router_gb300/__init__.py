"""GB300-native routed Mixture-of-Experts layer.

The compute path is the C-ABI library ``libmoe_gb300.so`` (hand-written CUDA
for sm_103a, sources in ``csrc/``); ``binding`` is its thin ctypes binding with
the same entry-point names, and ``synth`` draws seeded synthetic inputs.
Importing this package loads nothing: the library is loaded by the first
binding call, which raises if it is missing.
"""

__all__ = ["binding", "synth", "build"]
