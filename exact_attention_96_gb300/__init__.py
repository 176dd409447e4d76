"""Exact scaled-dot-product attention for GB300 (sm_103a).

The compute path is libfa_gb300.so (hand-written TMA / tcgen05 / TMEM kernels behind the C
ABI in include/fa.h).  This package only marshals arguments: ``abi`` mirrors the C entry
points one to one, ``attention`` wraps them for torch tensors, ``inputs`` draws the seeded
synthetic inputs, ``build`` compiles the library in-tree.
"""

from .attention import (forward, forward_fp8, forward_fp8_from_bf16, quantize_fp8,  # noqa: F401
                        forward_splitkv, backward, workspace_bytes, step_host, status_check)
