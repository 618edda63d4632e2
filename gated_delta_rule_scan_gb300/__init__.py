"""KDA / Gated DeltaNet gated delta-rule mixer for one GB300 (sm_103a).

Submodules:
  kda     ctypes binding of libkda (the C ABI in include/kda.h); loads the CUDA library
  mixer   whole-mixer calls that allocate buffers and run the entry points in stage order
  inputs  seeded synthetic workloads (no method arithmetic)
The binding is imported on first use so that ``inputs`` can be imported without the library.
"""

import importlib

__all__ = ["kda", "mixer", "inputs"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
