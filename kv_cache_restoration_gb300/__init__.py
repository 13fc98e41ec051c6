"""GB300-native KV-cache restoration from saved per-layer hidden states.

The computation lives in libhcr.so (C ABI: include/hcr.h), hand-written CUDA
for sm_103a.  Importing this package loads that library and fails loudly if
it has not been built; there is no CPU or PyTorch fallback.
"""
from . import binding  # noqa: F401  (raises ImportError if libhcr.so is missing)
from .binding import (  # noqa: F401
    HCR_OK, HcrError, hcr_cache_layout, hcr_check_device_error, hcr_create, hcr_destroy,
    hcr_last_error, hcr_model_dims, hcr_num_sms, hcr_restore, hcr_restore_prepare,
    hcr_restore_project, hcr_status_string, hcr_workspace_bytes)
from .restorer import Restorer, make_dims  # noqa: F401
