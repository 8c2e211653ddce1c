"""MiniMax-M3 MSA per-layer fused producer and paged-cache write for GB300 (sm_103a).

The producer runs in the CUDA library built from ``csrc/`` (C ABI in
``include/msa_producer.h``); ``binding`` marshals Python arguments into it and
``workloads`` makes seeded synthetic inputs.  Importing the package does not
load the library; the first call does, and raises if it is missing.
"""
from . import workloads  # noqa: F401

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in ("binding", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
