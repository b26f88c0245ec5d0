"""GB300-native (sm_103a) forward pass of a Flux-style MMDiT denoising step."""
