"""fp64 oracle of the acceptance step (the lossless accept / resample rule).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (page title, section):

* "Speculative decoding" guide (pigeon), *How it works*, steps 3-5: accept the
  drafted token with probability min(1, p/q); at the first rejection draw a
  replacement from norm(max(0, p - q)) and stop; if every draft survives, draw
  one bonus token from p at position gamma+1.  *Speed*: with greedy decoding
  the rule becomes "accept while argmax q = argmax p".  *When it breaks*:
  temperature and top-p are applied identically to p and q before the test.
* lattice-ai-eng "Speculative decoding" notes, the rule in words and the
  worked example (q(blue)=0.6, p(blue)=0.3, ratio 0.5, r=0.42 accepts, r=0.71
  rejects and resamples from the residual); the greedy collapse.
* "Build a Speculative Decoding Engine to Cut LLM Latency by 3x",
  *The Accept/Reject Mechanism*: the result record (accepted tokens,
  correction, n_accepted) and the numerical fallback to p when the residual
  mass is below 1e-8.

Readings where the pages leave a step open:

* Uniforms are inputs: u[i] (i < gamma) is the coin of the i-th ratio test and
  u[gamma] drives the single residual or bonus draw.
* A categorical draw is the inverse CDF in token-id order: the smallest id t
  whose cumulative weight exceeds u * (total weight).
* Top-p (the pages name it but do not define it): sort descending, ties by
  lower id; keep every token whose probability is >= the probability at the
  first position where the cumulative mass reaches top_p (ties at the
  threshold are all kept); renormalise.  Temperature is applied first.
* q(x) = 0 for a drafted token is a precondition violation (it cannot be
  drawn from q) and raises; the pages' epsilon guards are not reproduced.
* Greedy (T = 0): argmax with the lowest id on ties; q and u are ignored.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Decision margins inside which fp32 (device) and fp64 (oracle) arithmetic may
# legitimately disagree; such cases are counted, not failed.
RATIO_MARGIN = 1e-4
CDF_MARGIN = 1e-5
TOPP_MARGIN = 1e-5
RESIDUAL_FALLBACK = 1e-8


def softmax_t(z, temperature: float) -> np.ndarray:
    """p = softmax(z / T) in fp64 (lattice notes: softmax(logits / T))."""
    z = np.asarray(z, dtype=np.float64)
    if temperature <= 0:
        raise ValueError("softmax_t needs T > 0")
    s = z / np.float64(temperature)
    e = np.exp(s - s.max())
    return e / e.sum()


@dataclass
class NucleusInfo:
    kstar: int = -1          # sorted position where the cumulative mass reaches top_p
    tau: float = 0.0         # probability threshold: keep P >= tau
    kept: int = 0            # number of kept tokens
    boundary: bool = False   # cumulative mass within TOPP_MARGIN of top_p near k*


def nucleus(P: np.ndarray, top_p: float, margin: float = TOPP_MARGIN) -> tuple[np.ndarray, NucleusInfo]:
    """Top-p filter of one probability row, then renormalise.

    Reading of "top-p ... applied identically to p and q" (pigeon guide,
    *When it breaks*): the standard nucleus with the crossing token included
    and all ties at the threshold kept.
    """
    P = np.asarray(P, dtype=np.float64)
    info = NucleusInfo()
    if top_p >= 1.0:
        info.kept = int((P > 0).sum())
        return P.copy(), info
    if not top_p > 0.0:
        raise ValueError("top_p must be in (0, 1]")
    order = np.argsort(-P, kind="stable")       # descending, lower id first on ties
    c = np.cumsum(P[order])
    kstar = int(np.searchsorted(c, top_p, side="left"))   # first c_k >= top_p
    kstar = min(kstar, P.size - 1)
    tau = P[order[kstar]]
    keep = P >= tau
    out = np.where(keep, P, 0.0)
    out = out / out.sum()
    info.kstar, info.tau, info.kept = kstar, float(tau), int(keep.sum())
    near = abs(c[kstar] - top_p) < margin
    if kstar > 0:
        near = near or abs(c[kstar - 1] - top_p) < margin
    # two probabilities that are distinct in fp64 may tie in fp32 right at the
    # threshold; then the device keeps both and the oracle one
    if kstar + 1 < P.size:
        nxt = P[order[kstar + 1]]
        near = near or (tau > 0 and (tau - nxt) <= 1e-6 * tau and nxt < tau)
    info.boundary = bool(near)
    return out, info


def target_dist(z, temperature: float, top_p: float = 1.0, margin: float = TOPP_MARGIN):
    """The distribution a row of logits stands for: softmax(z/T), then top-p."""
    return nucleus(softmax_t(z, temperature), top_p, margin)


def argmax_lowest(z) -> int:
    """argmax with the lowest index on ties (np.argmax returns the first)."""
    return int(np.argmax(np.asarray(z, dtype=np.float64)))


@dataclass
class Draw:
    token: int
    boundary: bool


def inverse_cdf(w, u: float, margin: float = CDF_MARGIN) -> Draw:
    """Categorical draw from non-negative weights w with one uniform u in [0,1).

    Returns the smallest token id t with C_t = sum_{x<=t} w(x) > u * S,
    S = sum(w); a zero-weight token is never returned.  ``boundary`` is set
    when C_t or C_{t-1} lies within CDF_MARGIN * S of u * S.
    """
    w = np.asarray(w, dtype=np.float64)
    if np.any(w < 0):
        raise ValueError("negative weight")
    C = np.cumsum(w)
    S = C[-1]
    if not S > 0:
        raise ValueError("no mass to draw from")
    thr = np.float64(u) * S
    t = int(np.searchsorted(C, thr, side="right"))    # first C_t > thr
    if t >= w.size:                                    # u*S rounded up to S
        t = int(np.flatnonzero(w > 0)[-1])
    near = abs(C[t] - thr) < margin * S
    if t > 0:
        near = near or abs(C[t - 1] - thr) < margin * S
    return Draw(t, bool(near))


@dataclass
class AcceptResult:
    tokens: list                       # length gamma+1, -1 padded
    n_accepted: int
    emitted: int                       # the correction or bonus token
    bonus: bool                        # True when every draft was accepted
    ratio_boundary: bool = False       # some evaluated |u_i - min(1,p/q)| < RATIO_MARGIN
    cdf_boundary: bool = False         # the final draw sits on a CDF boundary
    topp_boundary: bool = False        # a nucleus used sits on its threshold
    fallback_boundary: bool = False    # residual mass near the 1e-8 fallback
    ratios: list = field(default_factory=list)

    @property
    def boundary(self) -> bool:
        return (self.ratio_boundary or self.cdf_boundary or self.topp_boundary
                or self.fallback_boundary)


def accept(z_target, q_draft, draft_tokens, uniforms, temperature: float,
           top_p: float = 1.0, margins: tuple | None = None) -> AcceptResult:
    """One sequence's verification outcome.

    z_target     [gamma+1][V] target logits (row i scores the token after
                 input i; rows 0..gamma-1 score x_1..x_gamma, row gamma is the
                 bonus position).
    q_draft      [gamma][V] the draft distributions the drafts were sampled
                 from, already after the same T / top-p (ignored for T = 0).
    draft_tokens [gamma] x_1..x_gamma.
    uniforms     [gamma+1] u_0..u_gamma in [0, 1) (ignored for T = 0).
    margins      (ratio, cdf, top_p) widths of the boundary flags; the
                 defaults cover fp32-vs-fp64 arithmetic on identical inputs.

    Follows pigeon *How it works* steps 3-5 and the lattice notes' rule.
    """
    z = np.asarray(z_target, dtype=np.float64)
    gamma = len(draft_tokens)
    if z.shape[0] != gamma + 1:
        raise ValueError("need gamma+1 target rows")
    V = z.shape[1]
    out = [-1] * (gamma + 1)

    if temperature == 0:
        # greedy: accept while the draft equals the target's argmax; on the
        # first mismatch emit the target's argmax; else the bonus argmax
        n = 0
        for i in range(gamma):
            a = argmax_lowest(z[i])
            if int(draft_tokens[i]) == a:
                out[i] = a
                n += 1
            else:
                out[i] = a
                return AcceptResult(out, n, a, False)
        a = argmax_lowest(z[gamma])
        out[gamma] = a
        return AcceptResult(out, gamma, a, True)

    rm, cm, tm = margins if margins is not None else (RATIO_MARGIN, CDF_MARGIN, TOPP_MARGIN)
    q = np.asarray(q_draft, dtype=np.float64)
    u = np.asarray(uniforms, dtype=np.float64)
    res = AcceptResult(out, 0, -1, False)
    for i in range(gamma):
        P, info = target_dist(z[i], temperature, top_p, tm)
        res.topp_boundary |= info.boundary
        x = int(draft_tokens[i])
        if not 0 <= x < V:
            raise ValueError("draft token out of range")
        if not q[i, x] > 0:
            raise ValueError("q(x) = 0 for a drafted token")
        a = min(1.0, P[x] / q[i, x])
        res.ratios.append(a)
        if abs(u[i] - a) < rm:
            res.ratio_boundary = True
        if u[i] < a:
            out[i] = x
            res.n_accepted += 1
            continue
        # first rejection: residual max(0, p - q) over the whole vocabulary
        r = np.maximum(P - q[i], 0.0)
        S = r.sum()
        if RESIDUAL_FALLBACK * 0.1 < S < RESIDUAL_FALLBACK * 10:
            res.fallback_boundary = True
        d = inverse_cdf(r if S > RESIDUAL_FALLBACK else P, u[gamma], cm)
        res.cdf_boundary = d.boundary
        out[i] = d.token
        res.emitted = d.token
        return res
    P, info = target_dist(z[gamma], temperature, top_p, tm)
    res.topp_boundary |= info.boundary
    d = inverse_cdf(P, u[gamma], cm)
    res.cdf_boundary = d.boundary
    out[gamma] = d.token
    res.emitted = d.token
    res.bonus = True
    return res


def draft_sample(z_draft, uniforms, temperature: float, top_p: float = 1.0):
    """The draft side of "applied identically": q = top-p(softmax(z/T)) per
    row, and a token drawn from q with one uniform by the same inverse CDF
    (T = 0: the argmax, q one-hot).  Returns (q [R][V] fp64, tokens [R],
    boundary [R])."""
    z = np.asarray(z_draft, dtype=np.float64)
    R, V = z.shape
    qs = np.zeros((R, V))
    toks = np.zeros(R, dtype=np.int64)
    bnd = np.zeros(R, dtype=bool)
    for r in range(R):
        if temperature == 0:
            a = argmax_lowest(z[r])
            qs[r, a] = 1.0
            toks[r] = a
            continue
        P, info = target_dist(z[r], temperature, top_p)
        d = inverse_cdf(P, float(uniforms[r]))
        qs[r], toks[r], bnd[r] = P, d.token, d.boundary or info.boundary
    return qs, toks, bnd
