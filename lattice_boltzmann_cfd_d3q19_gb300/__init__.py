"""GB300 (sm_103a) D3Q19 BGK lattice Boltzmann stream-collide library.

The compute path is liblbm.so (hand-written CUDA kernels behind the C ABI of include/lbm.h);
``binding`` exposes that ABI to Python under the same names, and ``workloads`` builds seeded
synthetic inputs.  Importing the package does not load the CUDA library; the first binding call
does, and fails loudly if it is missing.
"""
from . import workloads  # noqa: F401

__all__ = ["binding", "workloads", "build"]
