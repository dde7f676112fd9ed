"""libmoeep: MoE expert-parallel token dispatch and combine on one GB300 (sm_103a).

Submodules:
  moe_ep   -- ctypes binding of the C ABI in include/moe_ep.h (loads libmoeep.so;
              raises ImportError if it is not built -- there is no fallback)
  pipeline -- buffer allocation around one group + handle (torch memory only)
  synth    -- seeded synthetic workloads (no method arithmetic)
  build    -- nvcc build of libmoeep.so
The CUDA path is loaded on first use of ``moe_ep`` or ``pipeline``.
"""
import importlib

__all__ = ["moe_ep", "pipeline", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
