"""Block-diffusion speculative drafting (DFlash drafter + DDTree) on one GB300.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/dflash.h``); ``binding`` marshals PyTorch tensors into it.  Importing
this package does not load the library; the binding loads it on first use and
raises if it is missing.
"""
from .configs import WORKLOADS, DrafterShape, Workload  # noqa: F401
