"""GB300 (sm_103a) implementation of the Mamba-2 SSD selective scan, its
decode step and the Mamba-1 diagonal scan.

The compute path is the C-ABI library ``libssdscan.so`` (hand-written CUDA,
declared in ``include/ssd_scan.h``); :mod:`.binding` is the thin Python layer
over it (argument marshalling only). :mod:`.inputs` draws seeded synthetic
workloads. Importing the package does not load the CUDA library; the first
call into :mod:`.binding` does, and fails loudly if it has not been built.
"""
import importlib

__all__ = ["inputs", "binding", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
