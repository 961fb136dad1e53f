"""bit_kv_cache_rotate_b300: 4-bit rotated KV-cache decode attention for B300 (sm_103a)."""
