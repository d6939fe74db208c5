"""GB300 (sm_103a) three-segment INT2 KV cache: OSCAR's write and decode hot path.

Modules:
  build      compile the CUDA library in-tree (nvcc, sm_103a)
  binding    ctypes binding of include/oscar.h (argument marshalling only)
  calibrate  offline construction of R_K, R_V and clip thresholds
  synth      seeded synthetic inputs (no method arithmetic)
The binding is imported lazily so that the input generator and the offline
calibration can be used without the CUDA library.
"""

__all__ = ["build", "binding", "calibrate", "synth"]
