"""CPU oracle (test infrastructure only; see oracle.py's header)."""
from .oracle import *  # noqa: F401,F403
from .oracle import MoELayerOracle, ExpertSlotLRU  # noqa: F401
