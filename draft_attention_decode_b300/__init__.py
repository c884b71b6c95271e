"""Speculative-draft decode attention for B300 (sm_103a).

The compute path is the C-ABI library ``libdraft_attn.so`` (see
``include/draft_attn.h``); ``binding`` is its thin Python binding and
``workloads`` the seeded synthetic inputs.  Importing the package loads
nothing; ``binding`` loads the library and fails loudly if it is missing.
"""
__all__ = ["binding", "workloads", "build"]
