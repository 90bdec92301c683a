"""GB300 (sm_103a) decode step of hybrid Gated-DeltaNet / GQA / MoE transformers.

The compute lives in libhybrid.so (C ABI: include/hybrid.h), built by
``bandwidth_bound_hybrid_gb300.build.build()``.  ``capi`` is the ctypes
binding with the C names; ``model.HybridModel`` wraps a model and its cache.
"""
from . import capi  # noqa: F401

__all__ = ["capi"]
