"""GB300-native IO-aware exact attention (forward and backward), bf16, sm_103a."""
