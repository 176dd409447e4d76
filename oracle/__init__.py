"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls anything here, and this
package imports nothing from the product path.

What it computes is the plain definition of attention, written out in float64:

    S = scale * Q K^T   (+ causal mask: key j is hidden from query i when j > i)
    P = softmax(S) row by row
    O = P V
    LSE_i = m_i + ln(l_i),  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)

following "Flash Attention 原理与实践" §1.3 (the three-step standard computation),
"FlashAttention算子优化" §2 (the problem statement with scale = 1/sqrt(d)) and
"FlashAttention 与显存" §04 (S = QK^T, P = softmax(S), O = PV) and §09 (only O and the
per-row statistics are kept for the backward pass).

The backward pass is the analytic gradient of that definition (the pages give no
backward formulas; it is pinned by central finite differences and by torch.autograd
in the tests).

Modules
-------
attention       forward / backward definitions, whole tensors or sampled rows / heads
online_softmax  the streaming (running max, running sum) recurrence and the tiled
                forward in both loop orders the pages describe
io_model        FLOP and HBM-byte counters used by the pages' worked examples
philox          the counter-based generator behind the dropout mask

Parity status: every function here is pinned by tests under ``tests/`` (see
``tests/test_oracle_pins.py``) except the numbers of the online-softmax worked example
in "FlashAttention 与显存" §08, whose eight input scores are not printed: only its
invariant (blockwise == full-row) is checked, its printed values are parity unpinned.
"""

from . import attention, online_softmax, io_model, philox  # noqa: F401
