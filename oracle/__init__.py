"""CPU oracle for KV-cache restoration from hidden states.  TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import, call or execute anything in this package.  The CUDA library
(kv_cache_restoration_gb300) never imports it and shares no code with it.
"""
from . import restore, save, tiny_model  # noqa: F401
