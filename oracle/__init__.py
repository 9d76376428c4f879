"""Float64 CPU oracle (test infrastructure only; never imported by the product path)."""
from .sparse_mla_oracle import *  # noqa: F401,F403
from . import kv_append_oracle  # noqa: F401
from . import topk_select_oracle  # noqa: F401
