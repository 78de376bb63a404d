"""Single-GPU fused mixture-of-experts layer for GB300 (sm_103a).

The compute path lives in a C-ABI CUDA library (``include/moe.h``); the Python
functions in :mod:`.moe` only marshal arguments to it.  Importing this package
does not load the library; the first call does, and fails loudly when the
library is missing.
"""
