"""GB300-native (sm_103a) DFlash block-diffusion drafting step.

The hot path lives in libdflash.so (hand-written CUDA behind the C ABI of
include/dflash.h); ``binding`` exposes those calls under their C names and
``drafter`` adds weight packing, the paged KV cache and a small object
wrapper.  Nothing here computes the method on the host.
"""
from . import binding  # noqa: F401
from .binding import DflashError, load  # noqa: F401

__all__ = ["binding", "drafter", "DflashError", "load"]


def __getattr__(name):
    if name == "drafter":
        from . import drafter
        return drafter
    raise AttributeError(name)
