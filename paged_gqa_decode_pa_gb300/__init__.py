"""paged_gqa_decode_pa_gb300: paged grouped-query decode attention for GB300."""
