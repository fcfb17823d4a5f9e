"""Plain, slow CPU oracle for the mixed chunked-prefill + decode paged-attention step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product package (``mixed_chunked_prefill_gb300``) never imports
it, and this package imports nothing from the product.
"""

from .mixed_attn_ref import (  # noqa: F401
    PageTable,
    PagedKVStore,
    append,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    kv_head_of,
    merge_states,
    mixed_attention,
    new_token_slots,
    page_table_from_block_tables,
    segment_layout,
    visible_keys,
)
