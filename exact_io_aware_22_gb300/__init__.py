"""Exact IO-aware attention (FlashAttention-2 forward and backward) for GB300."""
