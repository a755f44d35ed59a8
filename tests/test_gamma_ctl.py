"""The library's host-side gamma controller (spec_gamma_ctl_*) against the
oracle (oracle.gamma): the depth rule on a grid of acceptance rates and
costs, and whole controllers driven by the same random pass records (several
slots, interleaved, window wrap-around, resets).  Host code only: runs
without a GPU.  Depth choices must be equal except where the oracle's two
best rates tie to 1e-12 (fp64 pow in C++ vs Python)."""
import numpy as np
import pytest

from oracle import gamma as G


@pytest.fixture(scope="module")
def sb():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verification_pass_gb300 import binding
    return binding


def _tied(alpha, gmin, gmax, td, tt, a, b):
    ra, rb = G.tokens_per_ms(alpha, a, td, tt), G.tokens_per_ms(alpha, b, td, tt)
    return abs(ra - rb) <= 1e-12 * max(ra, rb)


def test_depth_rule_matches_oracle(sb):
    for td, tt in ((2.0, 20.0), (0.5, 3.6), (5.0, 10.0), (0.0, 1.0)):
        for gmin, gmax in ((2, 8), (1, 16), (0, 4)):
            for alpha in np.concatenate([np.linspace(0, 1, 201), [0.999999, 1.0, 1.5]]):
                got = sb.spec_gamma_optimal(float(alpha), gmin, gmax, td, tt)
                ref = G.optimal_gamma(min(float(alpha), 1.0), gmin, gmax, td, tt)
                assert got == ref or _tied(min(alpha, 1.0), gmin, gmax, td, tt, got, ref), \
                    (alpha, gmin, gmax, td, tt, got, ref)


@pytest.mark.parametrize("window,min_records,td,tt", [(20, 5, 2.0, 20.0), (7, 3, 0.4, 3.6),
                                                      (1, 0, 1.0, 10.0)])
def test_controller_matches_oracle(sb, window, min_records, td, tt):
    rng = np.random.default_rng(window * 100 + min_records)
    slots = 6
    ctl = sb.GammaController(slots, 2, 8, 4, window, min_records, td, tt, 0.8)
    ref = [G.Controller(2, 8, 4, window, min_records, td, tt, 0.8) for _ in range(slots)]
    alpha_true = rng.uniform(0.2, 0.95, size=slots)
    for it in range(300):
        n = int(rng.integers(1, 9))
        s = rng.integers(0, slots, size=n)
        g = np.array([ref[k].gamma for k in s])
        # a slot listed twice uses its current depth for both entries
        a = np.array([min(gi, rng.geometric(1 - alpha_true[k]) - 1) for k, gi in zip(s, g)])
        got = ctl.step(s, g, a)
        exp = [ref[k].record(int(gi), int(ai)) for k, gi, ai in zip(s, g, a)]
        assert got == exp, (it, got, exp)
        if it % 50 == 49:
            k = int(rng.integers(0, slots))
            ctl.reset(k)
            ref[k] = G.Controller(2, 8, 4, window, min_records, td, tt, 0.8)
        for k in range(slots):
            al, gg, rr = ctl.state(k)
            assert abs(al - ref[k].alpha()) < 1e-12 and gg == ref[k].gamma and rr == len(ref[k].win)
    ctl.close()


def test_controller_rejects_bad_records(sb):
    ctl = sb.GammaController(2)
    with pytest.raises(sb.SpecError):
        ctl.step([0, 1], [4, 4], [2, 5])          # n_accepted > gamma_used
    assert ctl.state(1)[2] == 0 and ctl.state(0)[2] == 0   # nothing recorded
    with pytest.raises(sb.SpecError):
        ctl.step([2], [4], [1])                  # slot out of range
    with pytest.raises(sb.SpecError):
        sb.GammaController(2, gamma_min=5, gamma_max=3)
    ctl.close()
