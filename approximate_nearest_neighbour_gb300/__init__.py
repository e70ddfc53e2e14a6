"""Batched IVF-PQ search and exact flat k-NN on one GB300 (sm_103a).

The compute path is the C-ABI library ``libivfpq_gb300.so`` (declared in
``include/ivfpq.h``), built from ``csrc/`` by :func:`build.build_library`.
:mod:`.binding` is the thin ctypes layer over it (argument marshalling only);
it raises :class:`binding.LibraryMissing` when the library has not been built --
there is no CPU fallback. :mod:`.synthetic` holds the seeded input generators.
"""

from . import synthetic  # noqa: F401  (numpy only)

__all__ = ["synthetic", "binding", "build"]


def __getattr__(name):
    if name in ("binding", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
