"""CPU oracle for the W4A16 layer: test infrastructure only (see w4a16_oracle)."""
from .w4a16_oracle import *  # noqa: F401,F403
from . import w4a16_oracle as core  # noqa: F401
from . import fp8_oracle  # noqa: F401
