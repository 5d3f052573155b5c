"""GB300 (sm_103a) implementation of the GPTQ per-layer quantization path.

The compute lives in the CUDA library ``libgptq.so`` (C ABI in include/gptq.h);
``post_weight_quantization_gb300.gptq`` is its Python binding. Build the library with
``python -m post_weight_quantization_gb300.build``. Importing the binding without the
built library raises ImportError: there is no CPU fallback.
"""
import importlib

__all__ = ["gptq", "build"]


def __getattr__(name):
    if name in ("gptq", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
