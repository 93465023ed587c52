"""GroupQueryAttention over a shared, pre-allocated BNSH KV buffer on GB300.

The compute lives in libgqa.so (hand-written CUDA for sm_103a, C ABI in
include/gqa.h); this package is its Python binding.  PyTorch is used only for
device memory and streams."""
from ._binding import (EXPORTED, GQA_DTYPE_BF16, GQA_DTYPE_FP16, GQA_ERR_CUDA,  # noqa: F401
                       GQA_ERR_INVALID_ARGUMENT, GQA_ERR_KV_OVERFLOW, GQA_ERR_TIMEOUT,
                       GQA_ERR_UNSUPPORTED, GQA_OK, GqaError, gqa_check_device_status, gqa_decode_noalloc, gqa_dims_t,
                       gqa_forward, gqa_forward_host, gqa_status_string, gqa_workspace_size,
                       gqa_workspace_size_host, load_library, make_dims)
from .api import Workspace, forward, forward_host  # noqa: F401
