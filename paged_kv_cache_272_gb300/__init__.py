"""GB300-native paged KV-cache decode path.

The compute path is ``libpagedkv.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/pagedkv.h``); ``ops`` is its thin Python binding and
``block_pool`` wraps the native host block manager.  Importing this package loads
nothing; the binding loads the library on first use and raises if it is missing.
"""
__all__ = ["ops", "block_pool", "workloads"]
