"""CPU oracle for the FlashAttention-2 forward and backward passes -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything from this package.  The product path
(``exact_attention_24_gb300``) never imports it and never falls back to it.

The oracle is written from the definition of attention, in float64 NumPy:

* ``attention_ref`` / ``attention_ref_varlen`` -- the plain definition
  (explicit score matrix, max-shifted softmax, then ``@ V``, then the row
  log-sum-exp), following "FlashAttention -- for programmers, not
  researchers." (flash_attention_from_scratch.py), STAGE 1 (softmax) and
  STAGE 2 (standard attention), plus the scale and the ``L = m + log l``
  output of "Kernel visualization: Flash Attention 2", sections
  "Iteration j = 0" (scale after the dot product) and "Write the data back
  to HBM" (the L array).
* ``merge_partials`` -- STAGE 3's running-max / running-sum rescale applied
  to results computed over disjoint key ranges (the split-key merge).
* ``attention_tiled`` -- the tiled online-softmax loop of the same script's
  STAGE 3 (online softmax) and STAGE 4 (FlashAttention), used to pin the
  one-pass definition (block-size invariance) and to show that the
  no-rescale variant of STAGE 4 is wrong.

* ``attention_bwd_ref`` / ``attention_bwd_ref_varlen`` -- the gradients of
  ``sum(O * dO)`` from the plain definition (explicit P, the softmax
  derivative dS = P (dP - rowsum(dO O))), in the five contractions that
  "FlashAttention" (dao-ailab docs page), "Application in Backward Pass
  (5 MMAs)", lists.
* ``attention_bwd_recompute`` -- the same gradients by STAGE 5's route:
  P recomputed tile by tile from Q, K and the stored L.
* ``attention_bwd_sampled`` -- chosen rows of dQ and keys of dK, dV of one
  head, for checking full-size runs.

Every function here is pinned by ``tests/test_oracle.py`` and
``tests/test_oracle_bwd.py`` against closed forms, brute force in pure
Python, finite differences and ``torch`` CPU library routines.
"""

from .attention import (  # noqa: F401
    attention_ref,
    attention_ref_varlen,
    attention_tiled,
    attention_rows,
    merge_partials,
)
from .backward import (  # noqa: F401
    attention_bwd_magnitudes,
    attention_bwd_recompute,
    attention_bwd_ref,
    attention_bwd_ref_varlen,
    attention_bwd_sampled,
    forward_for_backward,
)
