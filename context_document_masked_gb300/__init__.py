"""Document-masked context-parallel attention for one GB300 (sm_103a).

Modules:
  fcp      ctypes binding of libfcp.so (include/fcp.h); raises on import if the
           library has not been built.
  session  CPAttention: one packed sequence, one plan, all shards on one GPU.
  build    nvcc build of libfcp.so.
"""
