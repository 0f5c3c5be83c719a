"""kvx for GB300: batched, descriptor-driven copies between mapped pinned host memory and HBM.

The compute path is ``libkvx.so`` (CUDA kernels for sm_103a plus a C++ host
engine behind the C ABI in ``include/kvx.h``, built by
``expert_host_block_gb300.build``); ``expert_host_block_gb300.kvx`` is its thin
ctypes binding.
"""
