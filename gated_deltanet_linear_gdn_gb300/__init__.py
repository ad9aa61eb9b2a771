"""GB300-native Gated DeltaNet layer hot path (conv update, fused decode step, chunked prefill)."""
