"""CPU oracle for the routed-expert MoE hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package.  See moe_oracle.py for the sources
and the readings it takes.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
from . import mx_oracle  # noqa: F401,E402
