"""GB300 block-scaled quantized linear kernels (sm_103a).

The compute path lives in the C-ABI shared library built from ``csrc/``
(``libr4q.so``); ``r4q`` is its thin ctypes binding. Importing this package
does not load the library; ``from block_scaled_precision_token_gb300 import r4q``
does, and raises if the library is missing.
"""

__all__ = ["r4q", "synth"]
