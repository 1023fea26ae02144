"""B300-native CSA2 sparse-attention decode step over an FP4 global KV cache.

* ``binding``   - ctypes binding of libcsa.so (the C ABI in include/csa.h)
* ``workloads`` - seeded synthetic inputs (random draws only)
* ``build``     - nvcc build of libcsa.so for sm_103a
"""
