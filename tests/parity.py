"""The token-parity bar shared by the GPU parity tests.

Emitted tokens and n_accepted must equal the oracle's on identical inputs.
A disagreement is excused only where the oracle flags the decision as lying
within its fp32-versus-fp64 margin, and excused disagreements must stay
below 0.1% of the cases.  Below 1000 cases that bound allows none, so the
bar is then zero.  The counts are printed (pytest -s shows them).
"""


def check(name: str, cases: int, near: int, excused: int, skipped: int = 0) -> None:
    """near = cases inside an oracle margin, excused = disagreements among
    them, skipped = end-to-end cases not graded because the decision lies
    within the logits tolerance of a boundary."""
    print(f"[parity] {name}: cases {cases}, in a margin {near}, excused {excused}, "
          f"end-to-end not graded {skipped}")
    if cases < 1000:
        assert excused == 0, (name, excused, cases)
    else:
        assert excused < 0.001 * cases, (name, excused, cases)
