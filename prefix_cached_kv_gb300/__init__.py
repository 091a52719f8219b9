"""prefix_cached_kv_gb300 -- attention of query rows over a resident shared-prefix KV cache on GB300.

The compute path is the CUDA library ``libpck.so`` (built from ``csrc/``); ``binding`` is a thin
ctypes layer that marshals torch tensors (device memory, streams) into its C ABI.
"""
