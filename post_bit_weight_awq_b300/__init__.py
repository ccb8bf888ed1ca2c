"""AWQ per-layer activation-aware scale search and INT4 packing for B300.

The compute path is libawq.so (hand-written CUDA for sm_103a behind a C ABI,
``include/awq.h``); ``capi`` is its ctypes binding and ``layer`` a one-call
wrapper that allocates with torch. Nothing here computes on the CPU.
"""
__all__ = ["capi", "layer", "multi"]


def __getattr__(name):
    if name in ("capi", "layer", "multi"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
