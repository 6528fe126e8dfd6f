"""CPU oracle for the single-GPU MoE layer forward (test infrastructure only).

The oracle is plain single-threaded C++ (``oracle.cpp``) compiled into
``liboracle.so`` and driven from here through ctypes with numpy buffers. Only the
test suite, the package smoke check and the benchmark's CPU-baseline leg use it;
the CUDA library never imports, links or calls anything in this directory.
"""

from .oracle import *  # noqa: F401,F403
