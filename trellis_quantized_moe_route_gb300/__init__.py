"""GB300 (sm_103a) fused MoE layer with bitshift-trellis-coded expert weights.

The layer lives in ``libtrellis_moe.so`` (hand-written CUDA behind the C ABI in
``include/trellis_moe.h``); ``binding`` is its thin ctypes wrapper and
``synth`` draws seeded synthetic inputs. Importing this package does not load
the library; the first binding call does, and raises if it is missing.
"""
__all__ = ["binding", "synth", "build"]
