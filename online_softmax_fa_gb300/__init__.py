"""GB300 (sm_103a) exact attention forward pass: O = softmax(scale*QK^T [+causal]) V
and LSE = m + log(l), behind a C-ABI library (``include/fa.h``).

``online_softmax_fa_gb300.fa`` is the thin ctypes binding; it loads the
in-tree CUDA library on first use and raises if it is missing.  Importing
this package does not load it.
"""
