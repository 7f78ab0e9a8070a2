"""Routed-expert MXFP4 mixture-of-experts layer for one GB300 GPU (sm_103a).

The compute lives in the CUDA library ``libmxfp4_moe.so`` (C ABI in
``include/mxfp4_moe.h``); ``moe`` is a thin ctypes binding with the same entry
points, ``synth`` draws seeded synthetic workloads.
"""
__all__ = ["moe", "synth"]
