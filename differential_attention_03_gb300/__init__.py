"""GB300-native multi-head differential-attention forward.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``libdiffattn.so``, built in-tree from ``csrc/``); ``binding`` is a
thin ctypes layer over it that only marshals arguments.  ``inputs`` draws the
seeded synthetic workloads.
"""

from .inputs import WORKLOADS, Workload  # noqa: F401


def __getattr__(name):
    # The binding loads the shared library on first use and fails loudly if it
    # is missing; importing the package for ``inputs`` alone needs no library.
    from . import binding
    return getattr(binding, name)
