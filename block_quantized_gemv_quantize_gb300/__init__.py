"""GB300 (sm_103a) small-M block-quantized GEMV and fused LM-head top-1.

The compute path is the C-ABI library ``libqgemv.so`` (hand-written CUDA
kernels, declared in ``include/qgemv.h``); ``ops`` re-exports its thin Python
binding.  Importing ``ops`` fails loudly when the library has not been built.
"""
from . import build  # noqa: F401


def __getattr__(name):
    if name == "ops":
        from . import _lib

        return _lib
    raise AttributeError(name)
