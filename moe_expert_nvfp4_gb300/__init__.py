"""GB300 (sm_103a) NVFP4 skinny-GEMM and MoE decode library.

The compute path lives in the C-ABI shared library ``libnvfp4moe.so`` built
from ``csrc/``; :mod:`moe_expert_nvfp4_gb300.ops` is its thin Python binding
(torch tensors in, pointers and sizes out).  :mod:`.synth` draws the seeded
synthetic inputs.  Importing this package does not load the library; the
first call into :mod:`.ops` does, and fails loudly if it is missing.
"""
__all__ = ["ops", "synth"]
