"""Seeded synthetic inputs for the MoE layer (shared by oracle tests, GPU tests and bench).

This module holds no arithmetic of the MoE method: it only produces input tensors
(activations, gate weights, expert weights) from a counter-based generator that
is bit-identical on the host (synth_host.c) and on the GPU (synth_dev.cu).
See synth_host.c for the exact definition.
"""

from .gen import (NORMAL, UNIFORM, normal_K, uniform_K, host_fill, dev_fill,  # noqa: F401
                  build_host, build_dev)
from .workloads import Workload, WORKLOADS, get  # noqa: F401
