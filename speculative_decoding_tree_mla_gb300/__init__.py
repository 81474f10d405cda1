"""Tree-verify MLA-absorb attention for GB300 (sm_103a).

The product is the C-ABI library ``libkdtv.so`` (declared in
``include/kdtv.h``); ``speculative_decoding_tree_mla_gb300.kdtv`` is a thin
ctypes binding over it.  Importing this package does not load the library;
the first call into the binding does, and raises if it was not built.
"""

__all__ = ["workloads", "kdtv"]
