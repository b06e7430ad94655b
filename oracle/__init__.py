"""Float64 CPU oracle of the PIC link step (test infrastructure only: see pic_oracle)."""
from .pic_oracle import *  # noqa: F401,F403
