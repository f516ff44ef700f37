"""B300-native (sm_103a) sparse Mixture-of-Experts FFN layer: a C-ABI CUDA
library (libmoe_b300.so, include/moe.h) and its thin ctypes binding."""

from . import moe  # noqa: F401
from .moe import (moe_capacity, moe_workspace_size, moe_route, moe_dispatch, moe_expert_ffn,  # noqa: F401
                  moe_combine, moe_layer_fwd, moe_layer_bwd, moe_check_error, make_config, config_of)
