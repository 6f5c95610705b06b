"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle's tests.

This package draws random numbers and packs them into the byte layouts the
library consumes. It holds none of the method's arithmetic: no dot product, no
activation, no fp8 decode, no argmax, no routing scan.
"""
from .decode_inputs import *  # noqa: F401,F403
