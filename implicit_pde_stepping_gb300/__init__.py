"""GB300-native batched pentadiagonal solves for semi-implicit PDE stepping.

The compute path is ``libpent.so`` (hand-written CUDA kernels for sm_103a
behind the C ABI of ``include/pent.h``); ``pent`` is its thin Python binding
and ``inputs`` the seeded synthetic workloads.  Importing the package does not
load the CUDA library; the first call into ``pent`` does, and fails loudly if
it has not been built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "pent", "build"]
