"""Pins of the oracle's K-SEQ multi-candidate verification at one position ("SpecTr:
Fast Speculative Decoding via Optimal Transport" page, section K-SEQ), CPU only.
The page writes p for the draft and q for the target; these tests, like the
oracle, write p for the TARGET and q for the DRAFT.

Each pin is fixed by the page or the mathematics and is chosen so that a
plausible slip fails one: the naive per-candidate rule (the page's
counterexample), a wrong root for rho*, a residual that forgets the direct
mass, the acceptance test with p and q swapped."""
import itertools

import numpy as np
import pytest

stats = pytest.importorskip("scipy.stats")


def test_pages_counterexample_naive_rule_overallocates(oracle_mod):
    """Draft always proposes A, target uniform on {A, B}, k = 2: accepting each
    candidate with min(1, p/q) gives A the mass 1/2 + 1/4 = 3/4 > p(A) = 1/2; K-SEQ's
    rho* = 1/2 / (1 - sqrt(1/2)) gives A exactly 1/2 and leaves B to the residual."""
    p, q, k = np.array([0.5, 0.5]), np.array([1.0, 0.0]), 2
    beta1 = oracle_mod.kseq_beta(p, q, 1.0)
    naive = (1 - (1 - beta1) ** k) / beta1 * min(q[0], p[0])
    assert abs(naive - 0.75) < 1e-15 and naive > p[0]
    A, pa, rho = oracle_mod.kseq_direct(p, q, k)
    assert abs(rho - 0.5 / (1 - np.sqrt(0.5))) < 1e-12
    assert abs(A[0] - 0.5) < 1e-12 and A[1] == 0.0 and abs(pa - 0.5) < 1e-12
    # both candidates rejected -> the residual is all on B
    assert oracle_mod.kseq_step(p, q, [0, 0], [0.99, 0.99], 0.2) == (1, -1)


def test_k1_is_the_single_candidate_rule(oracle_mod):
    """k = 1: rho* = 1, accept iff u q(x) < p(x), residual norm((p - q)+) -- the
    sampling oracle's first position with the same uniforms."""
    rng = np.random.default_rng(1)
    V, n = 12, 400
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    assert oracle_mod.kseq_rho(p, q, 1) == 1.0
    x = rng.choice(V, size=n, p=q)
    ua = rng.uniform(size=n)
    ur = rng.uniform(size=n)
    tgt = np.broadcast_to(np.log(p)[None, None], (n, 2, V)).astype(np.float32)
    drf = np.broadcast_to(np.log(q)[None, None], (n, 1, V)).astype(np.float32)
    # the sampling oracle normalises the float32 logits; use its rows for the K-SEQ side too
    pn = oracle_mod.normalise(tgt[0, 0].astype(np.float64), 1.0)
    qn = oracle_mod.normalise(drf[0, 0].astype(np.float64), 1.0)
    r = oracle_mod.verify(tgt, drf, x[:, None].astype(np.int32), np.ones(n, dtype=np.float32),
                          u_accept=ua[:, None], u_resid=np.stack([ur, ur], axis=1))
    for b in range(n):
        tok, idx = oracle_mod.kseq_step(pn, qn, [x[b]], [ua[b]], ur[b])
        assert (idx == 0) == (r.accepted_len[b] == 1)
        assert tok == r.out_tokens[b, r.accepted_len[b]] if idx < 0 else tok == x[b]


@pytest.mark.parametrize("k", [2, 3, 5])
def test_direct_mass_is_min_of_rho_q_and_p(oracle_mod, k):
    """At rho*, P_A = rho* beta(rho*) and A(x) = min(rho* q(x), p(x)) >= min(q(x), p(x))
    (the direct acceptance mass is never below the single candidate's)."""
    rng = np.random.default_rng(10 + k)
    for _ in range(20):
        V = rng.integers(2, 9)
        p = rng.dirichlet(np.ones(V) * rng.uniform(0.3, 3))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.3, 3))
        A, pa, rho = oracle_mod.kseq_direct(p, q, k)
        beta = oracle_mod.kseq_beta(p, q, rho)
        assert 1.0 <= rho <= k
        assert abs(pa - rho * beta) < 1e-9
        np.testing.assert_allclose(A, np.minimum(rho * q, p), atol=1e-9)
        assert (A >= np.minimum(q, p) - 1e-12).all() and (A <= p + 1e-12).all()


def test_fixed_rho_closed_form(oracle_mod):
    """If p(x) / rho <= q(x) for every x, beta(rho) = 1 / rho and the direct mass is
    [1 - (1 - 1/rho)^k] p(x), which tends to p as k grows (the page's special case)."""
    rng = np.random.default_rng(4)
    V, rho = 7, 2.0
    q = rng.dirichlet(np.ones(V) * 4)
    p = q * rng.uniform(0.6, 1.4, V)
    p /= p.sum()
    assert (p / rho <= q).all()
    beta = oracle_mod.kseq_beta(p, q, rho)
    assert abs(beta - 1 / rho) < 1e-15
    for k in (1, 3, 20):
        A = (1 - (1 - beta) ** k) / beta * np.minimum(q, p / rho)
        np.testing.assert_allclose(A, (1 - (1 - 1 / rho) ** k) * p, atol=1e-15)


@pytest.mark.parametrize("k", [2, 3])
def test_output_law_equals_target_exact_enumeration(oracle_mod, k):
    """Enumerate every candidate tuple (probability prod q(X_i)), try them in order with
    acceptance min(1, p / (rho* q)), then the normalised residual p - A: the emitted
    token's law must be p (within 1e-12), for drafters near and far from the target."""
    rng = np.random.default_rng(20 + k)
    V = 4
    for _ in range(10):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.2, 2))
        A, pa, rho = oracle_mod.kseq_direct(p, q, k)
        r = p - A
        assert (r >= -1e-12).all()
        res = r / r.sum() if r.sum() > 1e-300 else p
        a = np.where(q > 0, np.minimum(1.0, p / np.maximum(rho * q, 1e-300)), 0.0)
        law = np.zeros(V)
        for tup in itertools.product(range(V), repeat=k):
            w = np.prod(q[list(tup)])
            if w == 0.0:
                continue
            alive = 1.0
            for x in tup:
                law[x] += w * alive * a[x]
                alive *= 1.0 - a[x]
            law += w * alive * res
        np.testing.assert_allclose(law, p, atol=1e-12)


def test_output_law_chisquare_of_the_step(oracle_mod):
    """The whole step with uniforms: candidates drawn from q, 10^5 rounds, k = 3."""
    rng = np.random.default_rng(8)
    V, k, n = 6, 3, 100_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    counts = np.zeros(V, dtype=np.int64)
    cands = rng.choice(V, size=(n, k), p=q)
    us = rng.uniform(size=(n, k))
    ur = rng.uniform(size=n)
    for i in range(n):
        tok, _ = oracle_mod.kseq_step(p, q, cands[i], us[i], ur[i])
        counts[tok] += 1
    _, pval = stats.chisquare(counts, p * n)
    assert pval > 1e-3, (counts / n, p, pval)


def test_disjoint_supports_accept_nothing(oracle_mod):
    """beta = 0 (the page's special case): no candidate is accepted, the residual is p."""
    p = np.array([0.0, 0.0, 0.3, 0.7])
    q = np.array([0.5, 0.5, 0.0, 0.0])
    A, pa, _ = oracle_mod.kseq_direct(p, q, 3)
    assert pa == 0.0 and (A == 0).all()
    tok, idx = oracle_mod.kseq_step(p, q, [0, 1, 0], [0.0, 0.0, 0.0], 0.5)
    assert idx == -1 and tok == 3  # v = 0.5: past the 0.3 of token 2


# ---------------------------------------------------------------------------
# the batched entry: one position per row, Philox uniforms
# ---------------------------------------------------------------------------

def test_batched_equals_the_step_with_its_documented_uniforms(oracle_mod):
    rng = np.random.default_rng(31)
    B, K, V, seed = 64, 4, 20, 123
    tgt = (rng.normal(size=(B, V)) * 1.5).astype(np.float32)
    drf = (tgt + rng.normal(size=(B, V))).astype(np.float32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    nc = rng.integers(1, K + 1, B).astype(np.int32)
    cand = rng.integers(0, V, (B, K)).astype(np.int32)
    tok, acc, st = oracle_mod.kseq_verify(tgt, drf, cand, T, nc, seed=seed)
    assert (st == 0).all()
    for b in range(B):
        pn = oracle_mod.normalise(tgt[b].astype(np.float64), float(T[b]))
        qn = oracle_mod.normalise(drf[b].astype(np.float64), float(T[b]))
        u = [oracle_mod.uniform(seed, b, 1, 3 + i) for i in range(nc[b])]
        assert (tok[b], acc[b]) == oracle_mod.kseq_step(pn, qn, cand[b, : nc[b]], u, oracle_mod.uniform(seed, b, 1, 1))


def test_batched_one_candidate_is_the_sampling_verify(oracle_mod):
    """k = 1 with the same uniforms as the sampling oracle's position 1."""
    rng = np.random.default_rng(32)
    B, V, seed = 200, 15, 9
    tgt = rng.normal(size=(B, V)).astype(np.float32)
    drf = (tgt + rng.normal(size=(B, V)) * 0.8).astype(np.float32)
    T = np.ones(B, dtype=np.float32)
    x = rng.integers(0, V, (B, 1)).astype(np.int32)
    tok, acc, _ = oracle_mod.kseq_verify(tgt, drf, x, T, seed=seed)
    ua = np.array([[oracle_mod.uniform(seed, b, 1, 3)] for b in range(B)])
    ur = np.array([[oracle_mod.uniform(seed, b, 1, 1)] * 2 for b in range(B)])
    r = oracle_mod.verify(np.stack([tgt, tgt], axis=1), drf[:, None], x, T, u_accept=ua, u_resid=ur)
    assert ((acc == 0) == (r.accepted_len == 1)).all()
    assert (tok == np.where(r.accepted_len == 1, x[:, 0], r.out_tokens[:, 0])).all()


def test_batched_output_law_with_philox_uniforms(oracle_mod):
    """10^5 rows of one (p, q) pair, k = 3 candidates drawn from q: the emitted token ~ p."""
    rng = np.random.default_rng(33)
    B, K, V = 100_000, 3, 6
    lt, ld = rng.normal(size=V), rng.normal(size=V)
    tgt = np.broadcast_to(lt.astype(np.float32), (B, V)).copy()
    drf = np.broadcast_to(ld.astype(np.float32), (B, V)).copy()
    p = oracle_mod.normalise(lt.astype(np.float32).astype(np.float64), 1.0)
    q = oracle_mod.normalise(ld.astype(np.float32).astype(np.float64), 1.0)
    cand = rng.choice(V, size=(B, K), p=q).astype(np.int32)
    tok, _, _ = oracle_mod.kseq_verify(tgt, drf, cand, np.ones(B), seed=77)
    _, pval = stats.chisquare(np.bincount(tok, minlength=V), p * B)
    assert pval > 1e-3


def test_batched_status_bits(oracle_mod):
    rng = np.random.default_rng(34)
    B, K, V = 4, 2, 8
    tgt = rng.normal(size=(B, V)).astype(np.float32)
    tgt[2, 3] = np.inf
    cand = rng.integers(0, V, (B, K)).astype(np.int32)
    cand[1, 1] = -1
    tok, acc, st = oracle_mod.kseq_verify(tgt, tgt.copy(), cand, np.array([1, 1, 1, -1.0]), np.array([2, 2, 2, 2]),
                                          seed=1)
    assert st[0] == 0 and (st[1:] != 0).all() and (tok[1:] == -1).all() and (acc[1:] == -1).all()
