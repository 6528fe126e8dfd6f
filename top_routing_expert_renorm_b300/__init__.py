"""Single-GPU Mixture-of-Experts layer forward for B300 (sm_103a).

The layer (route -> dispatch -> expert FFNs -> combine) runs in hand-written CUDA
kernels inside libmoe.so, reached through a C ABI (include/moe.h). This package
is the thin Python binding over that ABI.
"""

from . import _capi  # noqa: F401
from .api import *  # noqa: F401,F403
from .api import MoeError, MoeConfig, MoeExpertWeights  # noqa: F401
from .moe_layer import MoELayer  # noqa: F401
