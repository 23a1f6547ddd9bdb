"""GB300-native paged KV-cache decode path.

The compute path lives in ``libpkv.so`` (hand-written sm_103a CUDA kernels and
a C++ host allocator behind a C ABI, declared in ``include/pkv.h``); ``pkv``
is its thin ctypes binding. Importing this package does not load the library;
the first call through ``pkv`` does, and raises if it is missing.
"""
