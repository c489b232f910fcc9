"""B300-native sparse MoE layer over Q4_K experts (sm_103a CUDA behind a C ABI)."""
