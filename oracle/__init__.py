"""OSCAR oracle -- TEST INFRASTRUCTURE, not part of the product.

A plain, slow, obviously correct CPU implementation (NumPy, float64 unless a
step's precision is fixed below) of what the three-segment INT2 KV-cache hot
path computes: rotation construction, clipping, INT2 quantisation, packing,
page allocation and three-segment decode attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  It shares no code with the CUDA
path and imports nothing from it.

Sources (web pages about OSCAR, "Offline Spectral Covariance-Aware Rotation"):
  [MTP] "Together AI Open-Sources OSCAR: An Attention-Aware 2-Bit KV Cache
        Quantization System for Long-Context LLM Serving" (MarkTechPost)
  [MS]  "TogetherAI开源OSCAR：超越 TurboQuant! 面向真实 Serving 的 2-bit KV
        Cache量化" (ModelScope community)
  [SP]  SourcePulse project card "OSCAR"

Parity status of each part is listed in the module docstrings.  Parts fixed by
a reading of the pages rather than by the pages themselves (the exact
quantiser convention, the calibration recipe, the byte layout) are pinned by
closed forms, invariants and brute force in ``tests/test_oracle_*.py``.
"""
from . import rotation, quant, layout, alloc, cache, attention  # noqa: F401
