"""B300-native Mamba-3 SSM layer recurrence: chunked prefill, decode step and
inter-chunk state passing as hand-written sm_103a CUDA kernels behind the C
ABI of ``include/m3.h`` (``libm3.so``).

``binding`` is the Python face of that ABI (ctypes, argument marshalling
only); ``synth`` draws seeded synthetic inputs; ``build`` compiles the library.
Importing the package does not load the library: the first call does, and
fails loudly if it is missing.
"""
from . import synth  # noqa: F401

__all__ = ["binding", "synth", "build"]


def __getattr__(name):
    if name in ("binding", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
