"""Simulated AllReduce on one GB300: N rank buffers in HBM reduced by
hand-written sm_103a kernels behind a C ABI (see include/ar.h)."""
