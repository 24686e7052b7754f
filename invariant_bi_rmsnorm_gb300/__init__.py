"""Batch-invariant forward kernels for LLM inference on GB300 (sm_103a)."""
