"""CPU oracle of the fused-MoE layer: test infrastructure, not product code.

Importable only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  It shares no code with the CUDA library.
"""
from . import codecs, moe_ref  # noqa: F401
