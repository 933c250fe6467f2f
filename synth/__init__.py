"""Seeded synthetic inputs shared by the oracle tests and the CUDA path (input generation only)."""
from .workloads import *  # noqa: F401,F403
