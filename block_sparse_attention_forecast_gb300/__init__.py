"""GB300-native forecast-driven block-sparse decode (SparDA).

The decode-step kernels live in libsparda.so (CUDA for sm_103a, C ABI in include/sparda.h);
``binding`` is its Python binding and ``step`` the decode-step driver that strings the calls
together on CUDA streams and graphs. The library is loaded on first use of any entry point;
if it is not built, that use raises ImportError (there is no fallback path).
"""
import importlib

_SUBMODULES = ("binding", "build", "step")


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(__name__ + "." + name)
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(importlib.import_module(__name__ + ".binding"), name)
