"""Padding-free packed bidirectional attention on GB300 (sm_103a).

Sequences are packed into one flat [num_tokens, heads, head_dim] buffer; each
sequence attends only to itself inside its cu_seqlens boundaries. The compute
lives in libpe.so (CUDA kernels behind the C ABI in include/pe.h); this
package is its thin Python binding plus the seeded synthetic workloads.
"""

from .binding import (  # noqa: F401
    PackedAttentionError,
    attention_workspace_bytes,
    load_library,
    pe_attention_kernel,
    pe_download_padded,
    pe_gather_packed,
    pe_flatten_packed_metadata,
    pe_geglu,
    pe_layernorm,
    pe_pack_document_ids,
    pe_pack_sequences,
    pe_packed_positions,
    pe_packed_attention_bwd,
    pe_packed_attention_bwd_local,
    pe_packed_attention_fwd,
    pe_packed_attention_fwd_local,
    pe_packed_attention_fwd_noalloc,
    pe_read_device_status,
    pe_read_noalloc_status,
    pe_rope_packed,
    pe_scatter_padded,
    pe_set_wait_limit_ns,
    pe_upload_packed,
)
