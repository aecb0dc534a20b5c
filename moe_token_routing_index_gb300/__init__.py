"""GB300-native routed-expert MoE forward.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``libmoe_gb300.so``, declared in ``include/moe.h``); ``binding``
marshals PyTorch tensors into it.  Importing this package does not load the
library; the first use of a binding name does, and raises if the library has
not been built (``python -m moe_token_routing_index_gb300.build``).
"""

import importlib

_SUBMODULES = ("binding", "build", "forward", "workloads")
__all__ = list(_SUBMODULES)


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    binding = importlib.import_module(f"{__name__}.binding")

    try:
        return getattr(binding, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
