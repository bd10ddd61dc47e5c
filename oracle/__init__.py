"""fp64 CPU oracle of the block-diffusion draft step (test infrastructure only)."""
from .dfl_oracle import *  # noqa: F401,F403
