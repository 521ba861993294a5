"""CPU oracle for the NVFP4 block-scaled linear layer (test infrastructure).

Only tests, the smoke check and the benchmark's CPU-baseline / reference legs
may import this package. The product path never does; it shares no code with
the CUDA kernels. See ``nvfp4_ref`` for what it computes and which passages of
the pages each function follows.
"""
from .nvfp4_ref import *  # noqa: F401,F403
