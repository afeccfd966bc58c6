"""fp64 CPU oracle (test infrastructure only; see ``dflash_oracle``)."""
from .dflash_oracle import *  # noqa: F401,F403
