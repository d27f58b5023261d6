"""GB300-native tree verify round: hand-written sm_103a CUDA kernels behind a C ABI.

Submodules:
  synth  -- seeded synthetic inputs (weights, caches, draft trees, uniforms)
"""
