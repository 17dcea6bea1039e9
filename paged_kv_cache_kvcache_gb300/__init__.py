"""libpagedattn: attention over a paged (block-table) bf16 KV cache on GB300 (sm_103a)."""
