"""MLA tree-verify attention for speculative decoding on GB300 (sm_103a).

The product is the C-ABI library libmlaverify.so (include/mla_verify.h):
an index/tree-mask builder kernel, the split-KV partial attention kernels
(tcgen05/TMEM tensor cores) and a log-sum-exp combine kernel; beside them (include/mla_decode_steps.h) greedy
tree acceptance, KV relocation and the fp8 paged indexer logits. This
package is its thin Python binding.
"""

from .binding import (  # noqa: F401
    D_QK,
    D_V,
    MLA_PARTIAL_PAIR,
    MLA_PARTIAL_QUAD,
    MLA_STATUS_BAD_INDPTR,
    MLA_STATUS_BAD_PARENT,
    MLA_STATUS_BAD_PREFIX,
    MLA_STATUS_BAD_SLOT,
    MLA_STATUS_CAPACITY,
    MLA_STATUS_EMPTY_ROW,
    MLA_STATUS_TIMEOUT,
    BoundCall,
    MlaError,
    alloc_workspace,
    bind_verify_attention_paged,
    library_path,
    load,
    mla_build_verify_meta,
    mla_fp8_indexer_logits,
    mla_kv_relocate,
    mla_tree_accept,
    mla_verify_attention,
    mla_verify_attention_anc,
    mla_verify_attention_paged,
    mla_verify_partial_paged,
    mla_verify_attention_noalloc,
    mla_verify_combine,
    mla_verify_init,
    mla_verify_noalloc_scratch_bytes,
    mla_verify_partial,
    mla_verify_reset_status,
    mla_verify_status_offset,
    mla_verify_version,
    mla_verify_workspace_bytes,
    partials,
    status_string,
    status_word,
)
from .device import DeviceInputs, to_device  # noqa: F401
