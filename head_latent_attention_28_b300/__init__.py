"""B300-native multi-head latent attention (MLA) decode.

A C-ABI CUDA library (libmla.so, declared in include/mla.h) with four calls
-- mla_cache_append, mla_absorb_query, mla_decode_paged, mla_absorb_output --
plus mla_decode_step (append, absorb and attend in one call), the prefill
pair mla_prefill_kv / mla_prefill_attention (attention over per-head keys and
values rebuilt from the latent cache), and this thin
Python binding with the same names.  PyTorch supplies device
memory and streams only; every step of the path runs in the library's
kernels.  Importing the package loads the library and fails loudly if it has
not been built.
"""

from ._lib import (  # noqa: F401
    LIB_PATH, MLA_BF16, MLA_ERR_BAD_INDEX, MLA_ERR_BAD_RECORD, MLA_ERR_CUDA, MLA_ERR_INVALID_ARG,
    MLA_ERR_TIMEOUT, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_F32, MLA_OK, PAGE_SIZE,
    SIGNATURES, MLAError, alloc_step_workspace, alloc_workspace, lib, load_library,
    mla_absorb_output, mla_absorb_output_merged, mla_absorb_output_merged_workspace_size,
    mla_absorb_query, mla_cache_append, mla_check_status, mla_merge_output_weights,
    mla_decode_item_cost, mla_decode_num_workers, mla_decode_paged, mla_decode_paged_noalloc,
    mla_decode_row_groups, mla_decode_split_plan, mla_decode_step, mla_decode_workspace_size,
    mla_prefill_attention, mla_prefill_kv, mla_prefill_kv_rows, mla_prefill_use_rebuild,
    mla_status_string, mla_test_force_splits, mla_test_set_wait_fault)

lib()  # load now: no silent fallback path exists
