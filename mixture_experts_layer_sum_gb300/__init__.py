"""Single-GPU Mixture-of-Experts layer for GB300 (sm_103a).

The product is the CUDA library libmoe_gb300.so (C ABI in include/moe.h).
`mixture_experts_layer_sum_gb300.moe` is its ctypes binding; other attributes
of this package resolve to it lazily, so building the library
(`python -m mixture_experts_layer_sum_gb300.build_ext`) works before it exists,
and any use of the layer without the library fails loudly.
"""
import importlib

_SUBMODULES = ("build_ext", "moe", "layer")


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    if name in _SUBMODULES:
        return importlib.import_module(__name__ + "." + name)
    mod = importlib.import_module(__name__ + ".moe")
    return getattr(mod, name)
