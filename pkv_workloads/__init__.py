"""Seeded synthetic inputs for paged-KV attention.

This package only draws random numbers and lays them out; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.
"""
from .gen import *  # noqa: F401,F403
