"""GB300-native multi-head differential-attention forward.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``libdiffattn.so``, built in-tree from ``csrc/`` by ``build.py``);
``binding`` is a thin ctypes layer over it that only marshals arguments.
``inputs`` draws the seeded synthetic workloads.
"""

import importlib

from .inputs import WORKLOADS, Workload  # noqa: F401

_API = ("lambda_init", "lambda_reparam", "diffattn_forward", "diffattn_v2_forward", "device_status",
        "debug_wait_timeout", "launch_count", "DiffAttnError")


def __getattr__(name):
    # The binding loads the shared library on first use and fails loudly if it
    # is missing; importing the package for ``inputs`` alone needs no library.
    if name in _API:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
