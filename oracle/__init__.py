"""CPU oracle of the Beam decoder-layer forward.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package entry's smoke check and the
benchmark's CPU-baseline leg may import this package. The CUDA path never imports, links or
calls it, and it shares no code with the CUDA path: its inputs come from the `synth` package or
from the tests themselves, never from a kernel.

Plain float64 NumPy, one step at a time, in the order the pages state the layer, with explicit
bfloat16 / FP8 rounding at the storage points (oracle/codecs.py).
"""
from . import codecs  # noqa: F401
from .beam_oracle import *  # noqa: F401,F403
