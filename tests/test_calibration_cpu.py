"""The library's latency-table calibration (host code, no GPU) against the
oracle: the same knee, coefficients and error to float64 rounding, and the
same float32 table bit for bit."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def bn():
    from tree_speculative_decoding_bastion_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


def close(x, y, scale):
    return abs(x - y) <= 1e-7 * max(1.0, scale)


CASES = [
    # (N grid, true a, b, c, knee, noise sigma, knee range)
    (np.array([1, 8, 16, 32, 64, 96, 128, 192, 256]), 5.0, 0.03, 0.1, 64, 0.0, (8, 200)),
    (np.arange(1, 257, 7), 12.0, 0.01, 0.25, 130, 0.3, (2, 250)),
    (np.arange(1, 257, 3), 3.0, 0.05, 0.0, 0, 0.05, (1, 256)),        # no hinge in the data
    (np.array([4, 4, 9, 9, 9, 30]), 1.0, 0.5, 0.0, 0, 0.01, (0, 40)),  # repeated N, knees below every N
    (np.array([10, 20, 10, 20]), 2.0, 1.0, 0.0, 0, 0.1, (0, 30)),      # two distinct N: every fit is a line
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("seed", range(3))
def test_fit_matches_oracle(bn, case, seed):
    N, a, b, c, knee, sigma, (lo, hi) = CASES[case]
    rng = np.random.default_rng(seed)
    t = a + b * N + c * np.maximum(0, N - knee) + rng.normal(0, sigma, N.size)
    got = bn.bastion_fit_verify_latency(N, t, lo, hi)
    want = oracle.fit_verify_latency(N, t, lo, hi)
    assert got[3] == want[3], (got, want)
    scale = float(np.abs(t).max())
    for g, w in zip(got[:3], want[:3]):
        assert close(g, w, scale), (got, want)
    assert abs(got[4] - want[4]) <= 1e-9 * max(1.0, want[4]) + 1e-12 * float(t @ t)


def test_table_matches_oracle_bit_for_bit(bn):
    rng = np.random.default_rng(9)
    for _ in range(20):
        a, b, c = rng.uniform(1, 10), rng.uniform(0, 0.1), rng.uniform(0, 0.5)
        knee = int(rng.integers(-5, 300))
        t_draft = rng.uniform(0, 3)
        n_max = int(rng.integers(1, 257))
        C, L_AR = bn.bastion_latency_table(a, b, c, knee, t_draft, n_max)
        Cw, Lw = oracle.latency_table(a, b, c, knee, t_draft, n_max)
        assert np.array_equal(C, Cw) and L_AR == Lw


def test_bad_input_is_refused(bn):
    with pytest.raises(bn.BastionError):
        bn.bastion_fit_verify_latency([5, 5, 5], [1.0, 2.0, 3.0], 0, 10)    # one distinct N
    with pytest.raises(bn.BastionError):
        bn.bastion_fit_verify_latency([1, 2], [1.0, 2.0], 0, 10)            # m < 3
    with pytest.raises(bn.BastionError):
        bn.bastion_fit_verify_latency([1, 2, 3], [1.0, float("nan"), 3.0], 0, 10)
    with pytest.raises(bn.BastionError):
        bn.bastion_fit_verify_latency([1, 2, 3], [1.0, 2.0, 3.0], 5, 4)
    with pytest.raises(bn.BastionError):
        bn.bastion_latency_table(1.0, 0.1, 0.0, 5, 0.0, 0)
