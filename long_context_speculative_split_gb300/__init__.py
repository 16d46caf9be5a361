"""GB300 (sm_103a) hot path of self-speculative decoding with a compressed draft KV cache.

The compute lives in libmgd.so (CUDA kernels behind the C ABI of include/mgd.h);
``mgd`` is its ctypes binding, ``ops`` allocates outputs/workspaces with torch
and calls the binding, ``workloads`` holds the seeded synthetic input
generators shared by the tests and the benchmark.
"""
from . import mgd  # noqa: F401
