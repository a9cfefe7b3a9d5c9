"""GB300-native fused attention forward + JVP (forward-mode flash attention).

The compute lives in the CUDA library built from ``csrc/`` (see ``build.py``);
this package holds the ctypes binding (``attention``), work/traffic counts
(``metrics``) and the seeded input generators shared with the tests
(``synth``).  Importing the package does not load the library; the first call
does, and raises if it has not been built.
"""

from .api import attention, device_status, fwd_dual, last_path  # noqa: F401

__all__ = ["attention", "fwd_dual", "device_status", "last_path"]
