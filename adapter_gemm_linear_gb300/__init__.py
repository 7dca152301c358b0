"""GB300-native multi-adapter LoRA linear layer.

out = x W^T + per-row (alpha_i/r_i) B_i (A_i x), with adapters in a paged
pool and rows reaching them by per-row id or by sorted segments.  The work is
done by liblora.so (C ABI in include/lora.h, CUDA kernels for sm_103a); this
package only binds it to PyTorch tensors and streams.
"""

from .api import (  # noqa: F401
    Int4Weight,
    Int8Weight,
    LinearCall,
    LoraError,
    LoraPool,
    abi_version,
    device_status,
    kernel_launches,
    linear_forward,
    pool_arena_bytes,
    pool_slot_bytes,
    segment_rows,
    status_string,
    arm_test_wait_timeout,
)
from .build import build  # noqa: F401
