"""GB300-native elu(x)+1 kernelized linear attention.

The compute path lives in the CUDA library ``liblinattn.so`` (sources under
``csrc/``, C-ABI declared in ``include/linattn.h``).  ``linattn`` is the thin
ctypes binding with the same entry-point names; ``workloads`` draws the seeded
synthetic inputs.  Importing this package does not load the library; the first
call through ``linattn`` does, and it raises if the library is missing.
"""
__all__ = ["linattn", "workloads"]
