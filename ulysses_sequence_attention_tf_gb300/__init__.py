"""GB300-native Ulysses sequence<->head relayout.

The compute path is the C-ABI library ``libtf_ulysses.so`` (hand-written sm_103a
CUDA, see ``csrc/``); ``binding`` is a thin ctypes layer over it.  Nothing here
has a CPU fallback: if the library is missing, the calls raise.
"""
import importlib

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
