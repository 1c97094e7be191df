"""CPU oracle for the 4-bit MoE expert-FFN layer (test infrastructure only;
see ``oracle/moe_oracle.py``)."""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
