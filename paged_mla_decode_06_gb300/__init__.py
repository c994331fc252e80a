"""Paged MLA decode for GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/mla_decode.h``); ``binding`` marshals PyTorch tensors into it.
Importing the package does not load the library: the first call does, and it
raises if the library is missing.
"""
__all__ = ["binding", "inputs"]
