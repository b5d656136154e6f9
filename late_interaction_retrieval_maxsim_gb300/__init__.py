"""GB300-native fused MaxSim (late-interaction scoring) -- placeholder, the
binding is added with the CUDA library."""
