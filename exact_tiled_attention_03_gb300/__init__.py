"""GB300-native exact FlashAttention forward (sm_103a CUDA behind a C ABI)."""
