"""Exact attention forward for GB300 (sm_103a).

``exact_io_aware_02_gb300.fa`` is the Python binding of the C-ABI library
``libfa_gb300.so`` (built in-tree by ``__graft_entry__.build()``); importing it
loads the library and fails loudly when it is missing.  ``inputs`` draws the
seeded synthetic tensors.  Nothing is imported eagerly here.
"""
