"""Fused scaled-dot-product attention for GB300 (sm_103a)."""
