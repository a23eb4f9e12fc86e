"""paged_kv_cache_213_gb300 -- paged decode attention for GB300 (sm_103a)."""
