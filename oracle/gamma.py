"""Oracle of the dynamic speculation-depth (gamma) controller.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source (page title, section): "Build a Speculative Decoding Engine to Cut
LLM Latency by 3x":

* *Speculation Depth Tuning and Tree Drafting*: tokens per target pass
  E(alpha, gamma) = (1 - alpha^(gamma+1)) / (1 - alpha) when each draft is
  accepted independently with probability alpha; the marginal gain of a
  deeper draft shrinks at low alpha; the controller follows the rolling
  acceptance rate of each sequence.
* *Dynamic Gamma Controller*: the depth is chosen to maximise tokens per
  second, not accepted tokens: the gamma in [gamma_min, gamma_max] (2..8 by
  default, 4 initially) maximising E(alpha, gamma) / (gamma * t_draft +
  t_target), with per-token draft and per-pass target latencies calibrated
  at start-up (2.0 ms and 20.0 ms in the page's setting); alpha is the
  acceptance rate over a window of the last 20 passes (0.80 assumed while
  the window is empty); no decision before 5 passes are recorded.
* *The Accept/Reject Mechanism* (the result record): a pass that accepts
  n of its gamma drafts records n accepted and gamma - n rejected.

Readings where the page leaves a step open:

* alpha over the window = (sum of accepted) / (sum of accepted + rejected),
  i.e. accepted drafts over drafted tokens (the page's estimator).
* At alpha >= 1 the expected tokens per pass are gamma + 1, the limit of the
  formula (every draft accepted plus the bonus token).
* Ties between depths go to the smaller gamma (the first maximum).
* The decision after each recorded pass uses that pass; the window keeps the
  last `window` passes of one slot (a sequence, or a group of sequences the
  caller pools, e.g. one content type).
"""
from __future__ import annotations

from collections import deque


def expected_tokens(alpha: float, gamma: int) -> float:
    """Tokens per target pass: the accepted drafts plus the correction or
    bonus token, (1 - alpha^(gamma+1)) / (1 - alpha)."""
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def tokens_per_ms(alpha: float, gamma: int, t_draft: float, t_target: float) -> float:
    return expected_tokens(alpha, gamma) / (gamma * t_draft + t_target)


def optimal_gamma(alpha: float, gamma_min: int, gamma_max: int, t_draft: float,
                  t_target: float) -> int:
    best, best_rate = gamma_min, -1.0
    for g in range(gamma_min, gamma_max + 1):
        r = tokens_per_ms(alpha, g, t_draft, t_target)
        if r > best_rate:
            best, best_rate = g, r
    return best


class Controller:
    """One slot's controller: a window of (accepted, rejected) per pass."""

    def __init__(self, gamma_min=2, gamma_max=8, gamma_init=4, window=20, min_records=5,
                 t_draft=2.0, t_target=20.0, alpha_prior=0.80):
        self.gmin, self.gmax = gamma_min, gamma_max
        self.gamma = gamma_init
        self.win = deque(maxlen=window)
        self.min_records = min_records
        self.t_draft, self.t_target = t_draft, t_target
        self.prior = alpha_prior

    def alpha(self) -> float:
        if not self.win:
            return self.prior
        acc = sum(a for a, _ in self.win)
        tot = sum(a + r for a, r in self.win)
        return acc / tot if tot > 0 else self.prior

    def record(self, gamma_used: int, n_accepted: int) -> int:
        if not 0 <= n_accepted <= gamma_used:
            raise ValueError("n_accepted outside [0, gamma]")
        self.win.append((n_accepted, gamma_used - n_accepted))
        if len(self.win) >= self.min_records:
            self.gamma = optimal_gamma(self.alpha(), self.gmin, self.gmax, self.t_draft,
                                       self.t_target)
        return self.gamma
