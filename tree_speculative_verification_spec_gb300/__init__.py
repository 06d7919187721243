"""GB300-native (sm_103a) tree speculative verification.

The product is libspectree.so, the CUDA library declared by include/spectree.h;
this package builds it (``build.build()``) and binds it (``_binding``): one
Python function per C entry point, same name, argument marshalling only.
"""
from ._binding import (SPEC_ATTN_AUTO, SPEC_ATTN_CUDA_CORE, SPEC_ATTN_NOALLOC_BYTES, SPEC_ATTN_TCGEN05, SPEC_BF16, SPEC_DEV_BAD_BLOCK,
                       SPEC_DEV_BAD_PATH, SPEC_DEV_BAD_TEMP, SPEC_DEV_BAD_TOKEN, SPEC_DEV_BAD_TREE, SPEC_DEV_CAPACITY, SPEC_DEV_TIMEOUT,
                       SPEC_ERR_CUDA, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_WORKSPACE, SPEC_F32,
                       SPEC_OK, SPEC_Q_PER_CHILD, SPEC_Q_PER_PARENT, SIGNATURES, SpecError, lib, spec_attention_workspace_size, spec_dsd_graph_keys, spec_dsd_optimal_k,
                       spec_dsd_select_k, spec_dsd_update, spec_kv_append, spec_kv_commit, spec_kv_commit_layers,
                       spec_philox_uniforms, spec_selftest_bounded_wait, spec_selftest_exp, spec_selftest_fx,
                       spec_selftest_resid, spec_tree_attention, spec_tree_expand_level, spec_tree_init,
                       spec_tree_mask_build, spec_tree_merge, spec_tree_verify_greedy,
                       spec_tree_verify_stochastic, spec_tree_attention_noalloc,
                       spec_verify_workspace_size, status_string, version, spec_dev_status_string, dev_status_names)
