"""GB300-native ReplaySSM cached SSM decode step.

The compute lives in ``libreplayssm.so`` (hand-written CUDA for sm_103a behind
a C ABI declared in ``include/replayssm.h``); ``_lib`` is the thin ctypes
binding with the same entry-point names.  ``synth`` draws seeded synthetic
workloads and ``traffic`` counts the algorithmic bytes of a step.

Importing the package does not load the CUDA library; the first call into
``_lib`` does, and raises if the library is missing (there is no CPU path).
"""

__all__ = ["synth", "traffic"]


def __getattr__(name):
    if name in ("synth", "traffic", "_lib", "build"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
