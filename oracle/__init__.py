"""CPU oracle of the MXFP4 routed-expert MoE layer — test infrastructure.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
it. Parity pins: see tests/test_oracle_pins.py.
"""
from .oracle import *  # noqa: F401,F403
