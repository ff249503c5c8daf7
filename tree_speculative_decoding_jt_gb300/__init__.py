"""GB300-native hot path of JetSpec-style tree speculative decoding.

The compute lives in libjt.so (hand-written CUDA for sm_103a behind the C ABI
of include/jt.h); this package holds its thin Python binding
(``binding``), the build script (``build``) and the seeded synthetic inputs
(``workloads``).
"""
from .binding import (  # noqa: F401
    EXPORTS, JT_DTYPE_BF16, JT_DTYPE_F32, JT_ERR_CUDA, JT_ERR_INVALID, JT_ERR_TIMEOUT, JT_ERR_UNSUPPORTED,
    JT_ERR_WORKSPACE, JT_OK, JT_OP_TREE_ATTN, JT_OP_TREE_BUILD, JT_OP_TREE_BUILD_MIXED,
    JT_OP_TREE_POLICY, JT_OP_TREE_TOPW, JT_OP_VERIFY_ACCEPT, JT_RULE_GREEDY, JT_RULE_MARGIN, JtError,
    PolicyParams, jt_check, jt_status_str, jt_tree_attn_paged, jt_tree_build, jt_tree_build_adaptive,
    jt_tree_build_mixed, jt_tree_build_noalloc, jt_tree_expand, jt_tree_expand_capped, jt_tree_policy,
    jt_tree_topw, jt_selftest_wait_timeout, jt_verify_accept, jt_verify_accept_stochastic, jt_version, jt_workspace_size,
    library_path, library_variant, load, policy_ceiling, policy_params, workspace)
