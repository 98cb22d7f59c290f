"""Simulated AllReduce on one GB300: N rank buffers in HBM reduced by
hand-written sm_103a kernels behind a C ABI (include/ar.h).

The C-ABI functions (``ar_allreduce``, ``ar_reduce_scatter``, ``ar_all_gather``,
``ar_bucketed_allreduce``, ...) are re-exported from ``.binding``, which loads
the compiled library on first use and raises if it is missing.  The input
generators in ``.workloads`` need no library.
"""
__version__ = "0.1.0"


def __getattr__(name):
    if name.startswith("ar_") or name in ("ArError", "check", "lib", "DTYPE", "OP", "ALGO", "STATUS", "MAX_RANKS"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
