"""GB300-native continuous-batching paged attention step.

The compute path lives in the C-ABI library `libkvpaged.so` (CUDA kernels for sm_103a);
`continuous_batching_paged_step_gb300.kvpaged` is its thin Python binding.  Importing
the binding fails loudly when the library has not been built.
"""
__all__ = ["kvpaged", "workloads"]
