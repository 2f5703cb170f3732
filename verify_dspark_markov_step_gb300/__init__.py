"""DSpark Markov drafting step and rejection-sampling verifier on one GB300.

The computation lives in the CUDA library built from ``csrc/`` (C ABI in
``include/dspark.h``); ``_lib`` binds it with ctypes. Submodules:

* ``build``      -- compiles ``_build/libdspark.so`` with nvcc for sm_103a
* ``_lib``       -- the binding (argument marshalling only)
* ``step``       -- one decode step (Markov loop + verification) on device tensors
* ``workloads``  -- seeded synthetic inputs
"""

__all__ = ["build", "workloads"]


def __getattr__(name):
    if name in ("markov_sample", "rejection_sample", "noise", "markov_workspace_bytes",
                "verify_workspace_bytes", "status_string", "DsparkError", "lib"):
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
