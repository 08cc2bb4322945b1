"""GB300-native (sm_103a) quantized Mixture-of-Experts expert path.

The compute lives in libqmoe.so (hand-written CUDA, C ABI declared in
include/qmoe.h); `binding` marshals torch tensors into it and `inputs` holds
the seeded synthetic workloads."""

__all__ = ["binding", "inputs", "build"]
