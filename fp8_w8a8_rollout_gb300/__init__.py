"""GB300-native FP8 W8A8 rollout linear path (binding filled in with the CUDA library)."""
