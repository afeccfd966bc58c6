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
    # ``drafter`` on first use; importing it by its full name keeps
    # ``from block_diffusion_drafter_context_gb300 import drafter`` from
    # re-entering this hook
    if name == "drafter":
        import importlib
        return importlib.import_module(__name__ + ".drafter")
    raise AttributeError(name)
