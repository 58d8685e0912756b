"""Paged-attention decode for GB300 (sm_103a)."""
