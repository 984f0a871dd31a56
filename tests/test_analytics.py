"""Acceptance analytics (host side) against the pages' printed numbers and the oracle."""
import numpy as np

from speculative_decoding_verification_20_gb300 import analytics as an


def test_fi_review_analysis_table(golden):
    """The (alpha, gamma) -> operations, speed table with c = c_hat = 0
    (tests/golden/expected_tokens_table.json)."""
    g = golden("expected_tokens_table.json")
    tol = g["printed_precision"]
    for row in g["rows"]:
        a, gm = row["alpha"], row["gamma"]
        assert abs(float(an.walltime_speedup(a, gm, 0.0)) - row["speed"]) <= tol
        assert abs(float(an.operations_increase(a, gm, 0.0)) - row["operations"]) <= tol
    b = g["also"]["bigram"]
    assert abs(float(an.walltime_speedup(b["alpha"], b["gamma"], 0.0)) - b["speedup_at_c0"]) <= tol
    lo, hi = g["also"]["alpha09_gamma7_tokens_range"]
    assert lo <= float(an.expected_tokens(0.9, 7)) <= hi


def test_corollary_and_optimal_gamma():
    """The page's corollary: gamma = 1 gives (1 + alpha) / (1 + c), an improvement
    whenever alpha > c; and its optimum for alpha = 0.9, c = 0.01 is gamma = 24."""
    for a, c in ((0.5, 0.1), (0.8, 0.05), (0.3, 0.29)):
        assert abs(float(an.walltime_speedup(a, 1, c)) - (1 + a) / (1 + c)) < 1e-15
        assert float(an.walltime_speedup(a, an.optimal_gamma(a, c), c)) >= (1 + a) / (1 + c)
    assert an.optimal_gamma(0.9, 0.01) == 24
    assert an.optimal_gamma(0.2, 0.5) == 1  # alpha < c: the first draft already costs more than it earns


def test_tau_with_equal_rates_is_the_geometric_closed_form():
    rng = np.random.default_rng(0)
    for _ in range(10):
        a, G = rng.uniform(0.05, 0.99), int(rng.integers(1, 12))
        tau = an.acceptance_length(np.full((1, G), a))[0]
        assert abs(tau - float(an.expected_tokens(a, G))) < 1e-12
    assert float(an.expected_tokens(1.0, 5)) == 6.0


def test_tau_from_the_steps_alpha_matches_the_mean_round_length(oracle_mod):
    """tau_b computed from the per-position alpha the oracle returns equals the mean
    number of tokens the oracle's rounds emit for those rows over many seeds."""
    rng = np.random.default_rng(5)
    B, G, V, seeds = 6, 4, 12, 4000
    tgt = (rng.normal(size=(B, G + 1, V)) * 1.5).astype(np.float32)
    drf = (tgt[:, :G] + rng.normal(size=(B, G, V)) * rng.uniform(0.2, 1.5, (B, 1, 1))).astype(np.float32)
    T = np.ones(B, dtype=np.float32)
    nd = np.array([4, 3, 2, 4, 1, 4], dtype=np.int32)
    tot = np.zeros(B)
    alpha = None
    for s in range(seeds):
        # drafts drawn from q for each seed (the law tau assumes)
        q = np.exp(drf / T[:, None, None])
        q /= q.sum(axis=2, keepdims=True)
        x = np.array([[rng.choice(V, p=q[b, i]) for i in range(G)] for b in range(B)], dtype=np.int32)
        r = oracle_mod.verify(tgt, drf, x, T, nd, seed=1000 + s)
        tot += r.accepted_len + 1
        alpha = r.alpha
    tau = an.acceptance_length(alpha, nd)
    mean = tot / seeds
    # the emitted count is at most gamma + 1: its standard deviation is below (gamma + 1) / 2
    assert (np.abs(mean - tau) < 4 * (nd + 1) / 2 / np.sqrt(seeds)).all(), (mean, tau)
    rates = an.position_rates(alpha, nd)
    assert np.isfinite(rates).all() and ((rates > 0) & (rates <= 1)).all()
