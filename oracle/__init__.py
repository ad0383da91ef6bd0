"""CPU oracle for the block-quantized GEMV path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg may import this package; the library (the CUDA path and its
Python binding) never does.  It shares no code with the CUDA path.
"""
from .oracle import *  # noqa: F401,F403
