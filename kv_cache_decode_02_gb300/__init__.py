"""kvattn for GB300: single-query split-KV decode attention (sm_103a CUDA kernels).

* ``kv_cache_decode_02_gb300.kvattn`` -- the Python binding of the C ABI declared in
  ``include/kvattn.h`` (loads ``_lib/libkvattn.so``; raises if it is not built).
* ``kv_cache_decode_02_gb300.inputs`` -- seeded synthetic inputs (no attention arithmetic).
* ``kv_cache_decode_02_gb300._build`` -- builds the library in-tree with nvcc.
"""
__version__ = "1.0.0"
