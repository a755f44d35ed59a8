"""fp64 oracle of constrained acceptance: one allowed-token set per logits
row, applied identically to the target and the draft logits.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source (page title, section):

* "Build a Speculative Decoding Engine to Cut LLM Latency by 3x", the
  interview question on constrained generation (JSON mode, grammar
  constraints): constrained generation puts a rejection mask on top of the
  token distribution; draft and target must both apply the same mask before
  their probabilities are computed (the constraint automaton runs in
  lockstep for both models); a mask applied on one side only, or in a
  different automaton state, makes the acceptance ratios wrong.

Readings where the page leaves a step open:

* A mask is one allowed-token set per logits row; the target row i and the
  draft row it is paired with carry the same set (the caller's automaton
  state after the same prefix).  Masking sets every disallowed logit to
  -inf, so after the temperature softmax (and top-p) a disallowed token has
  probability exactly 0 and the allowed tokens keep their relative weights;
  the acceptance rule then runs unchanged on the masked rows.
* A row that allows no token has no distribution to draw from: an error.
"""
from __future__ import annotations

import numpy as np


def apply_mask(z, allowed) -> np.ndarray:
    """Logits z [..][V] with every position where ``allowed`` is False set to
    -inf (fp64).  Raises when a row allows no token."""
    z = np.asarray(z, dtype=np.float64)
    a = np.asarray(allowed, dtype=bool)
    if a.shape != z.shape:
        raise ValueError("mask and logits shapes differ")
    if not a.any(axis=-1).all():
        raise ValueError("a row allows no token")
    return np.where(a, z, -np.inf)
