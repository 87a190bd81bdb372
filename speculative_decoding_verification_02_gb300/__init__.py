"""GB300-native speculative-decoding verification.

The verify-and-accept step that follows the target model's forward over k
drafted tokens: greedy prefix acceptance, lossless sampling acceptance with
residual resampling, tree verification, and the n-gram history drafter.
The work runs in hand-written sm_103a CUDA kernels behind the C ABI declared
in ``include/spec_verify.h`` (``libspecverify.so``); ``api`` is a thin ctypes
binding over it.  Importing the package loads nothing; ``api`` loads the
library on first use and raises if it has not been built.
"""

__all__ = ["api", "workloads"]


def __getattr__(name):
    if name in ("api", "workloads"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
