"""GB300-native InfiniGen speculative KV prefetch: the per-layer decode hot path."""
