"""CSA2 compressed sparse attention over a shared FP4 KV cache, for B300 (sm_103a).

The compute path is the CUDA library ``libcsa.so`` (C ABI in include/csa.h); ``binding`` marshals
torch tensors into its calls. ``synth`` holds the seeded synthetic-input generators.

Attributes of ``binding`` are reachable from the package (``csa.pack_fp4`` ...); the library is loaded
on first use and a missing build raises instead of falling back to anything else.
"""

import importlib

__all__ = ["binding", "synth", "build"]


def __getattr__(name):
    if name in ("binding", "synth", "build"):
        return importlib.import_module(f".{name}", __name__)
    mod = importlib.import_module(".binding", __name__)
    return getattr(mod, name)
