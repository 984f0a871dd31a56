"""Pins of the oracle's Gumbel-coupled (shared-noise) verification ("Speculative
decoding: the art of guessing well", section 共享噪声的采样), CPU only.

Each pin is a fact the page or the mathematics fixes, chosen so that a plausible
mistake fails one: independent instead of shared noise (match rate sum p*q),
the wrong sign in g = -log(-log u) (a biased law), a prefix rule off by one
(drafter invariance), filters not applied (the filtered law)."""
import numpy as np
import pytest

stats = pytest.importorskip("scipy.stats")


def _rows(logits, B, G):
    """The same logit row at every position of every sequence: [B, G, V] float32."""
    return np.broadcast_to(np.asarray(logits, dtype=np.float32)[None, None], (B, G, len(logits))).copy()


@pytest.mark.parametrize("T,k,p_top", [(1.0, None, None), (0.7, None, None), (1.0, 3, None), (1.3, None, 0.7)])
def test_target_token_follows_the_filtered_softmax(oracle_mod, T, k, p_top):
    """Gumbel-max: argmax_i(log p(i) + g_i) is a sample of p (section 共享噪声的采样,
    the exponential-clocks argument).  2 * 10^5 sequences, one row, V = 6."""
    rng = np.random.default_rng(7)
    V, B = 6, 200_000
    logits = rng.normal(size=V) * 1.5
    tgt = _rows(logits, B, 2)
    kk = None if k is None else np.full(B, k)
    pp = None if p_top is None else np.full(B, p_top)
    r = oracle_mod.gumbel_verify(tgt, np.zeros((B, 1), dtype=np.int32), np.full(B, T), None, kk, pp, seed=11)
    law = oracle_mod.normalise(logits.astype(np.float32).astype(np.float64), T, k or 0, p_top or 1.0)
    counts = np.bincount(r.target_tokens[:, 0], minlength=V)
    assert counts[law == 0].sum() == 0
    _, pval = stats.chisquare(counts[law > 0], law[law > 0] * B)
    assert pval > 1e-3, (counts / B, law, pval)
    # the second position uses independent noise: same law, different draws
    assert (r.target_tokens[:, 1] != r.target_tokens[:, 0]).mean() > 0.3


def test_emitted_tokens_do_not_depend_on_the_drafter(oracle_mod):
    """Drafter invariance: with the noise fixed, the round emits the target's own
    noise-driven tokens t_1..t_{n+1}, whatever the drafter; only n changes."""
    rng = np.random.default_rng(3)
    B, G, V = 256, 6, 40
    tgt = (rng.normal(size=(B, G + 1, V)) * 2).astype(np.float32)
    T = rng.uniform(0.5, 1.5, B)
    near = (tgt[:, :G] + rng.normal(size=(B, G, V)) * 0.3).astype(np.float32)
    far = (rng.normal(size=(B, G, V)) * 2).astype(np.float32)
    lens = []
    for drf in (near, far):
        x = oracle_mod.gumbel_draft(drf, T, seed=19)
        r = oracle_mod.gumbel_verify(tgt, x, T, seed=19)
        assert (r.status == 0).all()
        for b in range(B):
            n = r.accepted_len[b]
            assert (r.out_tokens[b, : n + 1] == r.target_tokens[b, : n + 1]).all()
            assert (r.out_tokens[b, :n] == x[b, :n]).all() and (n == G or x[b, n] != r.target_tokens[b, n])
            assert (r.out_tokens[b, n + 1:] == -1).all()
        lens.append(r.accepted_len.mean())
    assert lens[0] > lens[1] + 1.0  # the closer drafter matches more often
    # a drafter that proposes the target's own tokens is accepted in full
    r0 = oracle_mod.gumbel_verify(tgt, oracle_mod.gumbel_verify(tgt, np.zeros((B, G), dtype=np.int32), T,
                                                                seed=19).target_tokens[:, :G], T, seed=19)
    assert (r0.accepted_len == G).all()


def test_match_probability_is_the_pages_closed_form(oracle_mod):
    """P[argmax(log p + g) == argmax(log q + g)] = sum_j 1 / sum_i max(p_i/p_j, q_i/q_j)
    (section 共享噪声的采样), and (1 - TV) / (1 + TV) <= it <= 1 - TV."""
    rng = np.random.default_rng(5)
    V, B = 5, 400_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    closed = sum(1.0 / np.maximum(p / p[j], q / q[j]).sum() for j in range(V))
    tv = 0.5 * np.abs(p - q).sum()
    assert (1 - tv) / (1 + tv) <= closed <= 1 - tv
    x = oracle_mod.gumbel_draft(_rows(np.log(q), B, 1), np.ones(B), seed=23)
    r = oracle_mod.gumbel_verify(_rows(np.log(p), B, 2), x, np.ones(B), seed=23)
    rate = (x[:, 0] == r.target_tokens[:, 0]).mean()
    se = np.sqrt(closed * (1 - closed) / B)
    assert abs(rate - closed) < 4 * se, (rate, closed, se)
    assert abs(rate - (p * q).sum()) > 10 * se  # not the independent-noise rate
    assert abs(r.accepted_len.mean() - rate) < 1e-12  # gamma = 1: accepted iff the first tokens match


def test_greedy_is_the_argmax_prefix_rule(oracle_mod):
    """T = 0: no noise; the round is the greedy rule the sampling oracle also follows."""
    rng = np.random.default_rng(9)
    B, G, V = 128, 5, 30
    tgt = rng.normal(size=(B, G + 1, V)).astype(np.float32)
    drf = (tgt[:, :G] + rng.normal(size=(B, G, V)) * 0.5).astype(np.float32)
    x = drf.argmax(axis=2).astype(np.int32)
    r = oracle_mod.gumbel_verify(tgt, x, np.zeros(B), seed=1)
    s = oracle_mod.verify(tgt, drf, x, np.zeros(B), seed=1)
    assert (r.accepted_len == s.accepted_len).all() and (r.out_tokens == s.out_tokens).all()
    assert (r.target_tokens == tgt.argmax(axis=2)).all()


def test_invalid_rows_get_the_verify_status_bits(oracle_mod):
    rng = np.random.default_rng(2)
    B, G, V = 5, 3, 16
    tgt = rng.normal(size=(B, G + 1, V)).astype(np.float32)
    tgt[3, 1, 4] = np.nan
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    x[2, 0] = V
    T = np.array([1.0, -1.0, 1.0, 1.0, 1.0])
    nd = np.array([3, 3, 3, 3, 0])
    r = oracle_mod.gumbel_verify(tgt, x, T, nd, seed=4)
    s = oracle_mod.verify(tgt, tgt[:, :G].copy(), x, T, nd, seed=4)
    assert (r.status == s.status).all() and r.status[0] == 0 and (r.status[1:] != 0).all()
    assert (r.accepted_len[1:] == 0).all() and (r.out_tokens[1:] == -1).all()


def test_noise_layout(oracle_mod):
    """The token -> (Philox counter, word) mapping stated in the oracle's header."""
    seed = 0x1234_5678_9ABC
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    for b, pos, i in ((0, 1, 0), (3, 2, 5), (7, 4, 1023)):
        w = oracle_mod.philox4x32_10(np.array([b, pos, 2, i >> 2], dtype=np.uint32), key)[i & 3]
        assert oracle_mod.gumbel_uniform(seed, b, pos, i) == ((int(w) >> 8) + 0.5) / 2**24
