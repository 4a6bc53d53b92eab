"""Beam decoder-layer forward (decode and prefill) on one GB300: CUDA kernels for sm_103a
behind the C ABI of include/beam.h, with a thin ctypes binding (beam.py) and a host-side
layer/stack driver (stack.py). Importing the package does not load the library; the first
call does, and fails loudly if it was not built."""
from . import beam  # noqa: F401
