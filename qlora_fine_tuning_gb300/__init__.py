"""GB300-native QLoRA-adapted linear layer (sm_103a CUDA behind a C ABI).

The compute lives in ``libqlora.so`` (built from ``csrc/``); ``binding``
marshals numpy/torch arguments into its ``extern "C"`` entry points.  The
library is loaded lazily so that the input generator (``synth``) can be
imported on machines without the built library.
"""

__all__ = ["synth", "binding"]
