"""GB300 (sm_103a) DLRM sparse hot path.

The path -- embedding-bag forward, pairwise-interaction forward and backward,
embedding-bag backward with row-wise SGD -- runs in the CUDA library
``libdlrm_sparse.so`` behind the C ABI of ``include/dlrm_sparse.h``.  This
package is its thin Python binding (same names, torch tensors in, argument
marshalling only) plus the seeded workload generator used by the tests and
the benchmark.
"""
from ._native import (  # noqa: F401
    BF16, F16, F32, INT4, INTERACT_KERNEL_AUTO, INTERACT_KERNEL_CUDA_CORE, MAX_TABLES, DlrmError,
    dlrm_clear_error, dlrm_emb_bag_bwd_adagrad, dlrm_emb_bag_bwd_sgd, dlrm_emb_bag_bwd_sgd_atomic,
    dlrm_emb_bag_bwd_sgd_noalloc,
    dlrm_emb_bag_bwd_workspace_size, dlrm_emb_bag_coalesce, dlrm_emb_bag_fwd, dlrm_emb_bag_interact_fwd,
    dlrm_emb_bag_reduce_adagrad, dlrm_emb_bag_reduce_sgd, dlrm_emb_bag_sort_plan, dlrm_get_interact_kernel,
    dlrm_int4_row_bytes,
    dlrm_interact_bwd, dlrm_interact_fwd, dlrm_interact_width, dlrm_kernel_launch_count, dlrm_num_pairs,
    dlrm_profile_events, dlrm_quantize_int4, dlrm_read_error, dlrm_set_interact_kernel,
    dlrm_set_wait_test_hooks, library_path, load,
    status_string)
