"""GB300 (sm_103a) sparse-MLA decode over a paged FP8 latent KV cache.

The compute runs in libsparse_mla.so (CUDA, C ABI in include/sparse_mla.h);
this package is its thin PyTorch binding plus the seeded workload generator.
"""
from .api import (alloc_workspace, clear_errors, dims_of, make_dims, plan, plan_for, read_errors,  # noqa: F401
                  sparse_mla_combine, sparse_mla_decode, sparse_mla_gather_rows, sparse_mla_split,
                  sparse_mla_topk_select,
                  workspace_size)
