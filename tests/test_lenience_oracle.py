"""Pins of the oracle's lenient acceptance ("Fast Inference from Transformers via
Speculative Decoding" review page, section Lenience): a parameter l in [0, 1]
multiplies q(x) in the acceptance test, so a draft token is accepted iff
u * l * q(x) < p(x).  The page states two facts this must reproduce: no token is
emitted with more than 1/l times its target probability, and the acceptance
rate alpha rises as l falls.  The residual after a rejection is the page's
unchanged norm(max(0, p - q)) (the page changes only the test).
"""
import numpy as np
import pytest

from tests.test_oracle_pins import _log, _threshold


def _one(oracle_mod, lp, lq, x, u, v, l):
    """One sequence, gamma 1, float32 logits lp (both target rows) and lq, explicit uniforms."""
    tgt = np.stack([lp, lp])[None]
    return oracle_mod.verify(tgt, lq[None, None], np.array([[x]]), np.array([1.0]), u_accept=np.array([[u]]),
                             u_resid=np.array([[v, 0.5]]), all_positions=True, lenience=np.array([l]))


def _law(oracle_mod, p, q, l):
    """Black-box law of the first emitted token when x ~ q, from the oracle's acceptance
    region in u and its residual token as a function of v (found by bisection), the
    probability that the draft token is accepted, and the (p, q) the oracle holds for
    the float32 logits log p, log q (equal to p, q to about 1e-7)."""
    V = len(p)
    lp, lq = _log(p), _log(q)
    probe = oracle_mod.verify(np.stack([lp, lp])[None], lq[None, None], np.array([[0]]), np.array([1.0]), seed=0,
                              probs=True)
    p, q = probe.p_out[0, 0], probe.q_out[0, 0]
    resid, edges = np.zeros(V), [0.0]
    x0 = int(np.argmax(q))
    for y in range(V):
        up = _threshold(lambda v: _one(oracle_mod, lp, lq, x0, 0.999999, v, l).pos_token[0, 0] <= y)
        resid[y] = up - edges[-1]
        edges.append(up)
    law, accept = np.zeros(V), 0.0
    for x in range(V):
        if q[x] == 0:
            continue
        a = _threshold(lambda u: _one(oracle_mod, lp, lq, x, u, 0.5, l).pos_accept[0, 0] == 1)
        law[x] += q[x] * a
        law += q[x] * (1 - a) * resid
        accept += q[x] * a
    return law, accept, p, q


def _pair(seed, V):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(V) * 0.6)
    q = rng.dirichlet(np.ones(V) * 0.6)
    p[rng.integers(V)] = 0.0
    q[rng.integers(V)] = 0.0
    return p / p.sum(), q / q.sum()


def test_lenience_one_is_the_exact_rule(oracle_mod):
    rng = np.random.default_rng(5)
    B, G, V = 64, 4, 40
    t = rng.normal(size=(B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(size=(B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G))
    T = rng.choice([0.0, 0.7, 1.0], B)
    a = oracle_mod.verify(t, d, x, T, None, np.full(B, 10), np.full(B, 0.9), seed=9, all_positions=True)
    b = oracle_mod.verify(t, d, x, T, None, np.full(B, 10), np.full(B, 0.9), seed=9, all_positions=True,
                          lenience=np.ones(B))
    for f in ("accepted_len", "out_tokens", "alpha", "status", "pos_accept", "pos_token", "accept_margin",
              "resid_margin"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f), err_msg=f)


@pytest.mark.parametrize("seed,l", [(0, 0.5), (1, 0.3), (2, 0.1), (3, 0.8)])
def test_no_token_exceeds_one_over_l_times_its_probability(oracle_mod, seed, l):
    V = 6
    p, q = _pair(seed, V)
    law, accept, p, q = _law(oracle_mod, p, q, l)
    assert abs(law.sum() - 1.0) < 1e-9
    assert (law <= p / l + 1e-9).all(), (law, p / l)
    # the rule is lossy: the law moves off p toward q where q > p
    assert np.abs(law - p).max() > 1e-3
    # its value: min(q, p/l) from the draft, the rest from the residual norm(max(0, p - q))
    direct = np.where((l * q <= p) & (p > 0), q, np.where(p > 0, p / l, 0.0))
    r = np.maximum(p - q, 0.0)
    np.testing.assert_allclose(law, direct + (1 - direct.sum()) * r / r.sum(), atol=1e-9)
    # the oracle's alpha is the probability that the draft token is accepted
    p0, q0 = _pair(seed, V)
    tgt = np.stack([_log(p0), _log(p0)])[None]
    out = oracle_mod.verify(tgt, _log(q0)[None, None], np.array([[0]]), np.array([1.0]), seed=1,
                            lenience=np.array([l]))
    assert out.alpha[0, 0] == pytest.approx(accept, abs=1e-9)


def test_alpha_rises_as_lenience_falls(oracle_mod):
    rng = np.random.default_rng(11)
    B, V = 32, 300
    t = rng.normal(size=(B, 2, V)).astype(np.float32) * 2
    d = (t[:, :1] + rng.normal(size=(B, 1, V)) * 1.5).astype(np.float32)
    x = np.zeros((B, 1), np.int64)
    alphas = []
    for l in (1.0, 0.8, 0.5, 0.3, 0.1, 0.0):
        r = oracle_mod.verify(t, d, x, np.ones(B), seed=1, lenience=np.full(B, l))
        alphas.append(r.alpha[:, 0])
    alphas = np.array(alphas)
    assert (np.diff(alphas, axis=0) >= -1e-15).all()
    assert (alphas[-2] > alphas[0] + 0.05).all()
    # l = 1: sum_x min(p, q); l = 0: every draft token with p(x) > 0 passes (here all: no -inf)
    np.testing.assert_allclose(alphas[-1], 1.0, atol=1e-12)
    pq = oracle_mod.verify(t, d, x, np.ones(B), seed=1, probs=True)
    np.testing.assert_allclose(alphas[0], np.minimum(pq.p_out[:, 0], pq.q_out[:, 0]).sum(axis=1), atol=1e-12)


def test_zero_lenience_accepts_exactly_the_target_support(oracle_mod):
    p = np.array([0.5, 0.0, 0.3, 0.2, 0.0])
    q = np.array([0.1, 0.6, 0.1, 0.1, 0.1])
    for x in range(5):
        r = _one(oracle_mod, _log(p), _log(q), x, 0.999999, 0.5, 0.0)
        assert r.pos_accept[0, 0] == int(p[x] > 0)


def test_bad_lenience_is_flagged(oracle_mod):
    t = np.zeros((4, 2, 3), np.float32)
    d = np.zeros((4, 1, 3), np.float32)
    r = oracle_mod.verify(t, d, np.zeros((4, 1)), np.ones(4), seed=1,
                          lenience=np.array([1.0, -0.1, 1.5, np.nan], np.float32))
    assert list(r.status) == [0, oracle_mod.ST_BAD_LENIENCE, oracle_mod.ST_BAD_LENIENCE, oracle_mod.ST_BAD_LENIENCE]
    assert (r.out_tokens[1:] == -1).all() and (r.accepted_len[1:] == 0).all()


def test_chisquare_lenient_law(oracle_mod):
    """The oracle with its Philox uniforms samples the enumerated lenient law (10^5 rows)."""
    stats = pytest.importorskip("scipy.stats")
    V, B, l = 6, 100_000, 0.4
    p, q = _pair(21, V)
    law, _, _, _ = _law(oracle_mod, p, q, l)
    rng = np.random.default_rng(4)
    tgt = np.broadcast_to(np.stack([_log(p), _log(p)])[None], (B, 2, V)).copy()
    drf = np.broadcast_to(_log(q)[None, None], (B, 1, V)).copy()
    x = rng.choice(V, size=(B, 1), p=q)
    r = oracle_mod.verify(tgt, drf, x, np.ones(B), seed=8, lenience=np.full(B, l))
    counts = np.bincount(r.out_tokens[:, 0], minlength=V)
    keep = law > 0
    assert counts[~keep].sum() == 0
    _, pval = stats.chisquare(counts[keep], law[keep] / law[keep].sum() * B)
    assert pval > 1e-3, (counts / B, law, pval)
