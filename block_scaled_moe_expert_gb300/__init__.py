"""Block-scaled MoE experts forward for GB300 (sm_103a).

The compute path is the CUDA library built from csrc/ (libbsmoe.so, C ABI in
include/moe_experts.h); `binding` marshals torch tensors into it.
"""
from .binding import (MoeError, PreparedWeights, device_status, experts_forward, prepare_weights,  # noqa: F401
                      workspace_bytes, workspace_layout)
