"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .exl3_oracle import *  # noqa: F401,F403
from . import exl3_oracle  # noqa: F401
