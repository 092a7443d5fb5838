"""FP64 CPU oracle for causal blockwise ring attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package; the
product path (the CUDA library and its Python binding) never does, and this
package imports nothing from the product.

What it computes, in plain numpy float64, following the pages' definitions:

* ``attention``: naive full-matrix safe-softmax causal attention and its analytic
  backward (the tutorial "上下文并行", section "朴素 Ring Attention": the safe
  softmax equations and the per-chunk partial ``Softmax(Q K^T / sqrt(d)) V``; the
  InfiniTrain pull request "Feat: Context Parallel" #181, mode table row "p2p":
  single-pass online-softmax merge, backward by recomputing the probabilities),
  plus the (O, LSE) merge of two partial results, and one rank's share of the
  all-gather mode (pull request #181, mode table row "all_gather": local queries
  over the gathered K/V; K/V gradients summed over ranks by a ReduceScatter).
  Packed sequences: causal attention inside each document of a packed row
  (transformers pull request #50497: position ids restart mid-sequence and the
  mask is rebuilt for the packed documents).
* ``layouts``: the contiguous and zigzag (head-tail paired) token-to-rank maps
  (tutorial, section "Zig-Zag Ring Attention") and the all-to-all
  head<->sequence re-layout of the hierarchical a2a+p2p mode (pull request #181,
  mode table row "a2a+p2p"; tutorial, section "Ulysses CP").

Every function is pinned by CPU tests (``tests/test_oracle_*.py``) against closed
forms, invariants, finite differences, a library routine on the special cases it
covers, brute force on tiny inputs and the values the pages print.  No function
here is "parity unpinned".
"""
from . import attention, layouts  # noqa: F401
