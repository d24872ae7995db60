"""Paged KV cache decode path for GB300 (sm_103a): C-ABI library + thin binding."""
