"""Seeded synthetic inputs for paged decode attention.

This module serves both the CUDA path and the oracle. It holds none of the
method's arithmetic: it draws sequence lengths, physical block layouts and
normal values, places raw values in cache slots, and poisons every slot that
no sequence reads with NaN.
"""
from .configs import CONFIGS, Spec, get_config  # noqa: F401
from .gen import Workload, generate  # noqa: F401
