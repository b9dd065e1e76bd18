"""GB300-native low-precision MoE expert path (NVFP4 forward, MXFP8 backward)."""
