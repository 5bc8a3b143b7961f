"""GB300 paged KV cache: slot-mapped KV append, copy-on-write block copy and
paged decode attention (CUDA, sm_103a) behind a C ABI, plus a C++ host block
allocator.

The binding is in ``pagedkv`` (loaded on first use, raising if the library
has not been built); ``step`` drives one decode step through it; ``workloads``
draws seeded synthetic inputs.
"""
__all__ = ["pagedkv", "step", "workloads", "build"]
