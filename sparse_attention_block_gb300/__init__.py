"""GB300-native decode-time ICP block indexer.

Score fp8 index queries against a paged fp8 index-K cache into a float32
score plane (one column per B128 block), pick each (token, head) row's Top16
blocks with forced begin/end blocks, publish the lists as 33-word receive
rows, and merge per-shard lists -- every step in hand-written sm_103a CUDA
kernels behind the C ABI declared in ``include/icp.h``.

Submodules:
  ``icp``        -- the ctypes binding to ``libicp.so`` (raises if it is not built);
  ``workloads``  -- seeded synthetic inputs;
  ``build``      -- compiles the CUDA library in-tree.
"""
__version__ = "0.1.0"
