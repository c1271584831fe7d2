"""B300-native (sm_103a) selective-scan forward and decode state update.

The compute path is the CUDA library ``libssm.so`` built from ``csrc/``; this
package is a thin ctypes binding over its C ABI (``include/ssm.h``).  Importing
the package loads nothing; the library is loaded on first use and a missing or
unloadable library raises an error: there is no CPU fallback.
"""
from __future__ import annotations

__all__ = ["scan_fwd", "state_update"]


_BINDING_NAMES = ("scan_fwd", "state_update", "scan_fwd_workspace_size", "status_string",
                  "library", "ALGO_AUTO", "ALGO_CHANNEL", "ALGO_CHUNK", "SsmError")


def __getattr__(name):
    if name in _BINDING_NAMES:
        import importlib
        binding = importlib.import_module(__name__ + ".binding")
        return getattr(binding, name)
    raise AttributeError(name)
