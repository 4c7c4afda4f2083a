"""NVFP4 training linear layers on B300 (sm_103a).

The compute path is the C-ABI library ``libnvfp4.so`` built from ``csrc/``;
``binding`` marshals arguments into it.  Importing the package loads nothing;
the first call through ``binding`` loads the library and raises if it is
missing or if no CUDA device is present.
"""
__all__ = ["binding", "workloads"]
