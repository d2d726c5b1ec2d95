"""GB300-native confidence-driven variable-length verify step.

The step (confidence head + STS, survival-curve budget under a batch cap,
ragged compaction, speculative verify with accept/resample/bonus and commit)
runs in hand-written sm_103a CUDA kernels behind the C ABI declared in
``include/dspark.h`` (``libdspark.so``).  :mod:`.binding` is the thin ctypes
layer over that ABI; :mod:`.workloads` draws seeded synthetic inputs.
"""
__all__ = ["binding", "workloads"]
