"""GB300-native paged KV cache: paged decode attention, KV slot write and
copy-on-write block copy as CUDA kernels for sm_103a behind a C ABI
(``include/pa.h``), plus a host-side C++ block allocator.

``paged_kv_cache_142_gb300.ops`` is the thin Python binding over the C ABI
(argument marshalling only); ``workloads`` draws the seeded synthetic inputs.
The binding is imported lazily so that the input generators work on a host
without the built library.
"""
__all__ = ["ops", "workloads", "build"]
