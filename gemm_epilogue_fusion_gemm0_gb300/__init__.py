"""GB300-native (sm_103a) CODA chain: y = RMSNorm(x @ W0 + z, gamma) @ W1 as two
GEMM-epilogue programs, plus its data-gradient twin.

The compute lives in the C-ABI library ``libcoda.so`` (built from ``csrc/``);
``binding`` is a thin ctypes layer over it.  Importing the binding raises if
the library has not been built: there is no fallback path.
"""

import importlib

__all__ = ["synth", "binding"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
