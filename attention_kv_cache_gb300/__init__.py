"""Window-attention prompt-token scoring and top-k KV selection for GB300 (sm_103a).

Submodules:
  kvsel     ctypes binding of libkvsel.so (the C ABI in include/kvsel.h)
  pipeline  buffers plus the call order of the whole selection path
  synth     seeded synthetic workloads (shared input generator)
  build     nvcc build of libkvsel.so in-tree

``kvsel`` and ``pipeline`` load the compiled library on import and raise if
it is missing; ``synth`` and ``build`` need no GPU.
"""
