"""CPU models of the tensor-core kernels' barrier protocols, run under random
interleavings (see engine.py).  Test infrastructure; nothing in the library
imports them."""
