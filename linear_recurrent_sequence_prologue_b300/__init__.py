"""RetNet multi-scale retention on one B300: Python binding of libretention.so.

The compute path is the CUDA library (csrc/, C ABI in include/retention.h);
this package only marshals torch tensors into that ABI.
"""

from .api import (backward_plan, chunk_size, chunkwise, chunkwise_backward, decay_row_norm, force_path,
                  groupnorm, groupnorm_backward, matmul, msr_block, msr_block_plan, parallel, param_grads,
                  plan, rotate, selftest_timeout, status_string, step, sync_status)
from ._lib import (RET_BF16, RET_EINVAL, RET_ETIMEOUT, RET_EUNSUPPORTED, RET_EWORKSPACE, RET_F32,
                   RET_OK, RET_PATH_SIMT, RET_PATH_TC, RET_PATH_TC_CARRY, RET_PATH_TC_SINGLE, RetentionError,
                   load)

__all__ = [
    "chunkwise", "chunk_size", "chunkwise_backward", "backward_plan", "param_grads", "groupnorm",
    "groupnorm_backward", "decay_row_norm", "parallel", "step",
    "rotate", "plan", "sync_status", "selftest_timeout", "matmul", "msr_block", "msr_block_plan",
    "force_path", "status_string", "load", "RetentionError",
    "RET_OK", "RET_EINVAL", "RET_EUNSUPPORTED", "RET_ETIMEOUT", "RET_EWORKSPACE",
    "RET_F32", "RET_BF16", "RET_PATH_TC", "RET_PATH_SIMT", "RET_PATH_TC_SINGLE", "RET_PATH_TC_CARRY",
]
