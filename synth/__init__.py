"""Seeded synthetic inputs for the MXFP4 routed-expert MoE layer.

Inputs only: this package generates bytes and numbers with the workload's
distributions and shapes. It holds none of the layer's arithmetic; both the
CPU oracle and the CUDA library are fed from it.
"""
from .gen import *  # noqa: F401,F403
from .workloads import WORKLOADS, Workload  # noqa: F401
