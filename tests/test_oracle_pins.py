"""Pins of the fp64 oracle to what the pages and the mathematics fix (CPU only).

Each test names the passage it pins.  None of them re-types the oracle's own
formula: they use values printed on the pages, closed forms, identities that
the oracle does not compute itself, brute force over tiny vocabularies, and
black-box measurements of the oracle's decisions.
"""
import itertools
import math

import numpy as np
import pytest
from scipy import stats


def _log(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -np.inf).astype(np.float32)


def _one_position(oracle_mod, p_t, q_d, p_bonus=None, x=0, u=0.5, v=0.5):
    """Single sequence, gamma = 1, explicit uniforms; returns the oracle result."""
    V = len(p_t)
    p_bonus = p_t if p_bonus is None else p_bonus
    tgt = np.stack([_log(p_t), _log(p_bonus)])[None]
    drf = _log(q_d)[None, None]
    return oracle_mod.verify(tgt, drf, np.array([[x]]), np.array([1.0]), u_accept=np.array([[u]]),
                             u_resid=np.array([[v, 0.5]]), all_positions=True, probs=True)


# ---------------------------------------------------------------------------
# Worked examples printed on the SpecTr page (p = draft, q = target there)
# ---------------------------------------------------------------------------

def test_spectr_worked_example_overlap_and_residual(oracle_mod, golden):
    g = golden("spectr_worked_example.json")
    draft, target = np.array(g["draft"]), np.array(g["target"])
    # fp64 logits: the normalised rows reproduce the printed distributions exactly
    np.testing.assert_allclose(oracle_mod.normalise(np.log(target), 1.0), target, rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle_mod.normalise(np.log(draft), 1.0), draft, rtol=0, atol=1e-15)
    # the batched entry takes fp32 logits: log(p) rounded to fp32 moves p by < 1e-7
    r = _one_position(oracle_mod, target, draft)
    np.testing.assert_allclose(r.p_out[0, 0], target, rtol=0, atol=1e-7)
    np.testing.assert_allclose(r.q_out[0, 0], draft, rtol=0, atol=1e-7)
    # overlap = diagonal mass of the optimal coupling pi*
    pi = np.array(g["pi_star"])
    np.testing.assert_allclose(pi.sum(axis=1), draft, atol=1e-15)
    np.testing.assert_allclose(pi.sum(axis=0), target, atol=1e-15)
    assert abs(np.trace(pi) - g["diagonal_overlap"]) < 1e-15
    assert abs(r.alpha[0, 0] - g["diagonal_overlap"]) < 1e-7
    assert abs(np.minimum(target, draft).sum() - g["diagonal_overlap"]) < 1e-15
    # residual: measured from the oracle's draws over an evenly spaced grid of uniforms
    N = 4096
    us = (np.arange(N) + 0.5) / N
    counts = np.zeros(3)
    for v in us[:: N // 256]:
        rr = _one_position(oracle_mod, target, draft, x=0, u=0.999, v=v)  # draft token A rejected
        assert rr.accepted_len[0] == 0
        counts[rr.out_tokens[0, 0]] += 1
    np.testing.assert_allclose(counts / counts.sum(), g["residual_target"], atol=1e-12)


def test_spectr_two_candidate_single_acceptance(oracle_mod, golden):
    g = golden("spectr_two_candidate.json")
    r = _one_position(oracle_mod, np.array(g["target"]), np.array(g["draft"]))
    assert abs(r.alpha[0, 0] - g["single_candidate_acceptance"]) < 1e-7


def test_alpha_equals_one_minus_total_variation(oracle_mod):
    """alpha = sum min(p, q) = 1 - TV(p, q) = 1 - 1/2 sum |p - q| (art-of-guessing page, 投机采样)."""
    rng = np.random.default_rng(7)
    B, G, V = 16, 3, 50
    tgt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    drf = (tgt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    r = oracle_mod.verify(tgt, drf, rng.integers(0, V, (B, G)), np.ones(B), seed=3, probs=True)
    tv = 0.5 * np.abs(r.p_out[:, :G] - r.q_out).sum(axis=2)
    np.testing.assert_allclose(r.alpha, 1.0 - tv, atol=1e-14)


# ---------------------------------------------------------------------------
# Round length: E[#tokens] table, law of n, position-dependent tau
# ---------------------------------------------------------------------------

def _iid_alpha_batch(a, gamma, B, rng):
    """V = 3, p = (a, 1-a, 0), q = (a, 0, 1-a): sum min(p, q) = a at every position.
    Draft tokens are drawn from q (token 0 w.p. a, else token 2)."""
    p = np.array([a, 1 - a, 0.0])
    q = np.array([a, 0.0, 1 - a])
    tgt = np.broadcast_to(_log(p), (B, gamma + 1, 3)).copy()
    drf = np.broadcast_to(_log(q), (B, gamma, 3)).copy()
    x = np.where(rng.random((B, gamma)) < a, 0, 2)
    return tgt, drf, x


@pytest.mark.parametrize("row", range(6))
def test_expected_tokens_reproduces_printed_table(oracle_mod, golden, row):
    """E[#tokens] = (1 - a^(g+1)) / (1 - a); the printed Speed column (c = 0) equals it."""
    g = golden("expected_tokens_table.json")
    a, gamma, speed = (g["rows"][row][k] for k in ("alpha", "gamma", "speed"))
    closed = (1 - a ** (gamma + 1)) / (1 - a)
    assert abs(closed - speed) <= g["printed_precision"] + 1e-12
    assert abs((gamma + 1) / closed - g["rows"][row]["operations"]) <= g["printed_precision"] + 1e-12
    rng = np.random.default_rng(100 + row)
    B = 200_000
    tgt, drf, x = _iid_alpha_batch(a, gamma, B, rng)
    r = oracle_mod.verify(tgt, drf, x, np.ones(B), seed=11 + row)
    tokens = r.accepted_len + 1
    assert tokens.min() >= 1 and tokens.max() <= gamma + 1
    se = tokens.std() / math.sqrt(B)
    assert abs(tokens.mean() - closed) < 4 * se, (tokens.mean(), closed, se)
    np.testing.assert_allclose(r.alpha[:, :gamma], a, atol=1e-15)


def test_bigram_and_alpha09_examples(golden):
    g = golden("expected_tokens_table.json")["also"]
    bg = g["bigram"]
    assert abs((1 - bg["alpha"] ** (bg["gamma"] + 1)) / (1 - bg["alpha"]) - bg["speedup_at_c0"]) < 0.005
    lo, hi = g["alpha09_gamma7_tokens_range"]
    assert lo <= (1 - 0.9 ** 8) / 0.1 <= hi


def test_accepted_length_law_is_capped_geometric(oracle_mod):
    """P(n = k) = a^k (1 - a) for k < gamma and a^gamma at k = gamma (capped geometric)."""
    a, gamma, B = 0.7, 4, 300_000
    rng = np.random.default_rng(5)
    tgt, drf, x = _iid_alpha_batch(a, gamma, B, rng)
    r = oracle_mod.verify(tgt, drf, x, np.ones(B), seed=99)
    counts = np.bincount(r.accepted_len, minlength=gamma + 1)
    law = np.array([a ** k * (1 - a) for k in range(gamma)] + [a ** gamma])
    chi2, pval = stats.chisquare(counts, law * B)
    assert pval > 1e-3, (counts, law * B, pval)


def test_tau_with_position_dependent_alpha(oracle_mod):
    """tau = 1 + sum_k prod_{i<=k} a_i for fixed rows (art-of-guessing page, 我们能拿到多少 token)."""
    alphas = [0.9, 0.75, 0.6, 0.4, 0.2]
    gamma, B = len(alphas), 200_000
    rng = np.random.default_rng(17)
    tgt = np.zeros((B, gamma + 1, 3), np.float32)
    drf = np.zeros((B, gamma, 3), np.float32)
    x = np.zeros((B, gamma), np.int64)
    for i, a in enumerate(alphas):
        tgt[:, i] = _log([a, 1 - a, 0.0])
        drf[:, i] = _log([a, 0.0, 1 - a])
        x[:, i] = np.where(rng.random(B) < a, 0, 2)
    tgt[:, gamma] = _log([1 / 3] * 3)
    r = oracle_mod.verify(tgt, drf, x, np.ones(B), seed=123)
    tau = 1 + sum(np.prod(alphas[: k + 1]) for k in range(gamma))
    tokens = r.accepted_len + 1
    assert abs(tokens.mean() - tau) < 4 * tokens.std() / math.sqrt(B)


# ---------------------------------------------------------------------------
# Exactness: the output marginal equals p for any q
# ---------------------------------------------------------------------------

def _threshold(f, lo=0.0, hi=1.0, iters=60):
    """Smallest u in [lo, hi] where the monotone predicate f switches from True to False."""
    if not f(lo):
        return lo
    if f(hi):
        return hi
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if f(mid):
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _measured_output_law(oracle_mod, p, q, p_next):
    """Black-box law of the first emitted token when x ~ q: the oracle's acceptance
    region in u and its residual token as a function of v are measured by bisection."""
    V = len(p)
    law = np.zeros(V)
    # residual token as a function of v (monotone): breakpoints by bisection
    tok_at = lambda v: _one_position(oracle_mod, p, q, p_next, x=int(np.argmax(q)), u=0.999999, v=v)
    resid = np.zeros(V)
    edges = [0.0]
    for y in range(V):
        up = _threshold(lambda v: tok_at(v).pos_token[0, 0] <= y)
        resid[y] = up - edges[-1]
        edges.append(up)
    for x in range(V):
        if q[x] == 0:
            continue
        acc = lambda u: _one_position(oracle_mod, p, q, p_next, x=x, u=u).pos_accept[0, 0] == 1
        a = _threshold(acc)
        law[x] += q[x] * a
        law += q[x] * (1 - a) * resid
    return law


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_enumeration_marginal_equals_target(oracle_mod, seed):
    """Leviathan et al. A.1 / SpecTr (1): P(output = x) = p(x) for any q.  V <= 8, with zeros."""
    rng = np.random.default_rng(seed)
    V = 5 + seed
    p = rng.dirichlet(np.ones(V) * 0.7)
    q = rng.dirichlet(np.ones(V) * 0.7)
    p[rng.integers(V)] = 0.0
    q[rng.integers(V)] = 0.0
    p /= p.sum()
    q /= q.sum()
    law = _measured_output_law(oracle_mod, p, q, p)
    np.testing.assert_allclose(law, p, atol=1e-9)


def test_exact_enumeration_second_position(oracle_mod):
    """gamma = 2: given the first draft token was accepted, the second emitted token ~ p_2."""
    rng = np.random.default_rng(42)
    V = 6
    p1, q1, p2, q2, p3 = (rng.dirichlet(np.ones(V)) for _ in range(5))
    x1 = int(np.argmax(np.minimum(p1, q1)))
    law = np.zeros(V)
    def run(x2, u2, v2):
        tgt = np.stack([_log(p1), _log(p2), _log(p3)])[None]
        drf = np.stack([_log(q1), _log(q2)])[None]
        return oracle_mod.verify(tgt, drf, np.array([[x1, x2]]), np.array([1.0]),
                                 u_accept=np.array([[1e-9, u2]]), u_resid=np.array([[0.5, v2, 0.5]]),
                                 all_positions=True)
    r0 = run(0, 0.5, 0.5)
    assert r0.pos_accept[0, 0] == 1
    resid = np.zeros(V)
    prev = 0.0
    for y in range(V):
        up = _threshold(lambda v: run(int(np.argmax(q2)), 0.999999, v).pos_token[0, 1] <= y)
        resid[y] = up - prev
        prev = up
    for x2 in range(V):
        a = _threshold(lambda u: run(x2, u, 0.5).pos_accept[0, 1] == 1)
        law[x2] += q2[x2] * a
        law += q2[x2] * (1 - a) * resid
    np.testing.assert_allclose(law, p2, atol=1e-9)


def test_bonus_token_law_is_next_target_distribution(oracle_mod):
    """All gamma drafts accepted: the extra token is drawn from p_{gamma+1} itself
    (Algorithm 1 step 4 keeps p' = p_{n+1} when n = gamma; q_{gamma+1} is treated as zero)."""
    rng = np.random.default_rng(77)
    V = 7
    p1, q1, p2 = (rng.dirichlet(np.ones(V)) for _ in range(3))
    x1 = int(np.argmax(np.minimum(p1, q1)))
    def run(v):
        tgt = np.stack([_log(p1), _log(p2)])[None]
        drf = _log(q1)[None, None]
        return oracle_mod.verify(tgt, drf, np.array([[x1]]), np.array([1.0]), u_accept=np.array([[1e-9]]),
                                 u_resid=np.array([[0.5, v]]))
    assert run(0.5).accepted_len[0] == 1
    law, prev = np.zeros(V), 0.0
    for y in range(V):
        up = _threshold(lambda v: run(v).out_tokens[0, 1] <= y)
        law[y], prev = up - prev, up
    np.testing.assert_allclose(law, p2, atol=1e-7)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_chisquare_marginal_million_draws(oracle_mod, seed):
    """10^6 sequences, V = 8, gamma = 1, x ~ q: first emitted token ~ p (chi-square)."""
    rng = np.random.default_rng(1000 + seed)
    V, B = 8, 1_000_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    tgt = np.broadcast_to(np.stack([_log(p), _log(p)]), (B, 2, V)).copy()
    drf = np.broadcast_to(_log(q)[None], (B, 1, V)).copy()
    x = rng.choice(V, size=(B, 1), p=q)
    r = oracle_mod.verify(tgt, drf, x, np.ones(B), seed=seed)
    first = r.out_tokens[:, 0]
    counts = np.bincount(first, minlength=V)
    _, pval = stats.chisquare(counts, p * B)
    assert pval > 1e-3, (counts / B, p, pval)


# ---------------------------------------------------------------------------
# Greedy reduction, normalisation, filters
# ---------------------------------------------------------------------------

def test_greedy_is_longest_argmax_prefix_plus_target_token(oracle_mod):
    """T = 0: keep the longest prefix with x_i = argmax p_i, then append argmax p_{n+1}."""
    rng = np.random.default_rng(3)
    B, G, V = 400, 5, 12
    tgt = rng.integers(-3, 4, (B, G + 1, V)).astype(np.float32)  # many ties
    drf = rng.integers(-3, 4, (B, G, V)).astype(np.float32)
    am = tgt.argmax(axis=2)  # numpy: first index of the maximum
    x = np.where(rng.random((B, G)) < 0.7, am[:, :G], rng.integers(0, V, (B, G)))
    r = oracle_mod.verify(tgt, drf, x, np.zeros(B), seed=5)
    for b in range(B):
        n = 0
        while n < G and x[b, n] == am[b, n]:
            n += 1
        assert r.accepted_len[b] == n
        assert list(r.out_tokens[b, :n]) == list(x[b, :n])
        assert r.out_tokens[b, n] == am[b, n]
        assert all(r.out_tokens[b, n + 1:] == -1)
        np.testing.assert_array_equal(r.alpha[b], (am[b, :G] == drf[b].argmax(axis=1)).astype(float))


def test_softmax_ratios_and_mass(oracle_mod):
    rng = np.random.default_rng(8)
    lg = rng.normal(0, 3, 300)
    for T in (0.3, 1.0, 2.5):
        p = oracle_mod.normalise(lg, T)
        assert abs(p.sum() - 1) < 1e-14
        i, j = 17, 123
        assert abs(np.log(p[i] / p[j]) - (lg[i] - lg[j]) / T) < 1e-12


def test_argmax_one_hot_lowest_id(oracle_mod):
    lg = np.array([1.0, 5.0, 2.0, 5.0, -np.inf])
    np.testing.assert_array_equal(oracle_mod.normalise(lg, 0.0), [0, 1, 0, 0, 0])


def test_filter_identities(oracle_mod):
    rng = np.random.default_rng(9)
    lg = rng.normal(0, 2, 64)
    base = oracle_mod.normalise(lg, 0.7)
    np.testing.assert_array_equal(oracle_mod.normalise(lg, 0.7, top_k=64), base)
    np.testing.assert_array_equal(oracle_mod.normalise(lg, 0.7, top_k=0), base)
    np.testing.assert_array_equal(oracle_mod.normalise(lg, 0.7, top_p=1.0), base)


@pytest.mark.parametrize("seed", range(4))
def test_filters_brute_force_small_vocab(oracle_mod, seed):
    """top-k: the k most probable (lower id on ties); top-p: a smallest set reaching top_p,
    made of the most probable tokens; both renormalised.  Brute force over all subsets."""
    rng = np.random.default_rng(seed)
    V = 7
    lg = rng.integers(-4, 3, V).astype(np.float64) * 0.5  # exact ties on purpose
    T = 0.9
    soft = np.exp(lg / T - (lg / T).max())
    soft /= soft.sum()
    key = lambda i: (-soft[i], i)
    for k in range(1, V + 1):
        got = oracle_mod.normalise(lg, T, top_k=k)
        kept = set(np.nonzero(got)[0])
        assert kept == set(sorted(range(V), key=key)[:k])
        np.testing.assert_allclose(got[list(kept)], soft[list(kept)] / soft[list(kept)].sum(), rtol=1e-13)
    for tp in (0.05, 0.3, 0.5, 0.77, 0.95, 0.999):
        got = oracle_mod.normalise(lg, T, top_p=tp)
        kept = set(np.nonzero(got)[0])
        best = min(len(s) for n in range(1, V + 1) for s in itertools.combinations(range(V), n)
                   if soft[list(s)].sum() >= tp)
        assert len(kept) == best, (tp, kept, best)
        worst_kept = max(kept, key=key)
        assert all(key(j) > key(worst_kept) for j in set(range(V)) - kept)
        np.testing.assert_allclose(got[list(kept)], soft[list(kept)] / soft[list(kept)].sum(), rtol=1e-13)
    # top-k then top-p: the nucleus is taken inside the renormalised top-k set
    for k in (2, 4):
        for tp in (0.4, 0.8):
            got = oracle_mod.normalise(lg, T, top_k=k, top_p=tp)
            topk = sorted(range(V), key=key)[:k]
            sk = soft[topk] / soft[topk].sum()
            n = int(np.searchsorted(np.cumsum(sk), tp - 1e-15) + 1)
            assert set(np.nonzero(got)[0]) == set(topk[:n])


# ---------------------------------------------------------------------------
# Invariants and argument handling
# ---------------------------------------------------------------------------

def test_round_length_invariant_and_layout(oracle_mod):
    rng = np.random.default_rng(21)
    B, G, V = 300, 6, 40
    tgt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    drf = (tgt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    nd = rng.integers(1, G + 1, B)
    r = oracle_mod.verify(tgt, drf, rng.integers(0, V, (B, G)), np.full(B, 0.8), num_draft=nd, seed=4)
    assert (r.accepted_len >= 0).all() and (r.accepted_len <= nd).all()
    for b in range(B):
        n = r.accepted_len[b]
        assert 0 <= r.out_tokens[b, n] < V
        assert (r.out_tokens[b, n + 1:] == -1).all()
        assert (r.alpha[b, nd[b]:] == 0).all()


def test_status_bits(oracle_mod):
    B, G, V = 6, 2, 5
    tgt = np.zeros((B, G + 1, V), np.float32)
    drf = np.zeros((B, G, V), np.float32)
    x = np.zeros((B, G), np.int32)
    T = np.ones(B, np.float32)
    tk = np.zeros(B, np.int32)
    tp = np.ones(B, np.float32)
    T[0] = -1.0
    tk[1] = -3
    tp[2] = 0.0
    x[3, 1] = V
    tgt[4, 1, 2] = np.nan
    tgt[5, 0, :] = -np.inf
    r = oracle_mod.verify(tgt, drf, x, T, top_k=tk, top_p=tp, seed=1)
    m = oracle_mod
    assert list(r.status) == [m.ST_BAD_TEMPERATURE, m.ST_BAD_TOP_K, m.ST_BAD_TOP_P, m.ST_BAD_DRAFT_TOKEN,
                              m.ST_NONFINITE, m.ST_NONFINITE]
    assert (r.out_tokens == -1).all() and (r.accepted_len == 0).all()
    nd = np.array([0, 1, 2, 3, 1, 1])
    r = oracle_mod.verify(np.zeros((B, G + 1, V), np.float32), drf, np.zeros((B, G)), np.ones(B),
                          num_draft=nd, seed=1)
    assert list(r.status[:4]) == [m.ST_BAD_NUM_DRAFT, 0, 0, m.ST_BAD_NUM_DRAFT]


# ---------------------------------------------------------------------------
# Philox4x32-10: statistical pins only (no published vector stored here)
# ---------------------------------------------------------------------------

def test_philox_uniforms_are_uniform_and_independent(oracle_mod):
    ua, ur = oracle_mod.philox_uniforms(seed=2024, B=1 << 15, G=7)
    u = np.concatenate([ua.ravel(), ur.ravel()])
    assert u.min() > 0 and u.max() < 1
    # on the 24-bit grid
    np.testing.assert_array_equal((u * 2 ** 24 - 0.5) % 1.0, 0.0)
    counts = np.histogram(u, bins=256, range=(0, 1))[0]
    assert stats.chisquare(counts).pvalue > 1e-3
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # neighbouring counters are uncorrelated
    assert abs(np.corrcoef(ua[:, 0], ua[:, 1])[0, 1]) < 0.02
    assert abs(np.corrcoef(ua[:, 0], ur[:, 0])[0, 1]) < 0.02


def test_philox_bits_balanced_and_distinct(oracle_mod):
    outs = np.array([oracle_mod.philox4x32_10([i, 7, 1, 0], [0x12345678, 0x9ABCDEF0]) for i in range(4096)],
                    dtype=np.uint32)
    bits = ((outs[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.abs(bits - 0.5).max() < 0.05
    assert len({tuple(o) for o in outs}) == len(outs)
    a = oracle_mod.philox4x32_10([1, 2, 3, 4], [5, 6])
    b = oracle_mod.philox4x32_10([1, 2, 3, 4], [5, 7])
    assert bin(int(a[0]) ^ int(b[0])).count("1") > 4
