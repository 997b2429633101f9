"""kvattn for GB300: split-KV decode attention (sm_103a CUDA kernels) over f16, Q8_0 and
Q4_0 KV caches -- contiguous, through a compact cell plan, or a resident window merged with
a pinned host tail -- for one query token per sequence or a few draft tokens (causal).

* ``kv_cache_decode_02_gb300.kvattn`` -- the Python binding of the C ABI declared in
  ``include/kvattn.h`` (loads ``_lib/libkvattn.so``; raises if it is not built).
* ``kv_cache_decode_02_gb300.inputs`` -- seeded synthetic inputs (no attention arithmetic).
* ``kv_cache_decode_02_gb300._build`` -- builds the library in-tree with nvcc.
"""
__version__ = "1.0.0"
